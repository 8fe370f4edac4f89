"""Benchmark: gate-level time-based power analysis on GB300.

One step = one pass of the whole hot path over the loaded workload: event-count
partition -> fused dynamic + leakage power kernel -> final reduction (one
``pa_run`` on the loaded per-pin layout; nothing is prepared for it outside the
step). Default workload: the very large skewed configuration (5M gates, 64
cells with 1-4 inputs and 8x8 LUTs, 100k cycles at 1 ns, 1B events with
Zipf(1.1) gate activity), seeded synthetic inputs.

Printed (rank 0, one JSON line):
  value    events/s over all ranks, inputs resident in HBM, timed with CUDA
           events on the library's stream over the timed steps (after a
           warm-up of at least --warmup steps and --warmup-seconds), max over
           ranks; the median step beside it
  roofline the fused kernel's algorithmic bytes per launch / its mean duration
           (CUDA events recorded on its stream inside pa_run) against the
           measured HBM copy bandwidth; the median and the whole pass beside it
  banded_layout  the cycle-banded layout beside the timed pass: its build time
           (pa_build_bands, once per trace and clock) and runs on it (the
           re-run figure of a trace analysed at several voltages or window
           ends), reported, not the value
  e2e      same metric through the public API with host buffers: per step the
           events are copied from pinned host memory (pa_load_events, with
           device-side validation), the pass runs, and the waveform and counts
           come back to the host; a one-shot run streams the trace through
           the device (pa_run_stream), or loads it and runs the unbanded kernel,
           or loads it and builds the banded layout first: all are timed and the
           fastest is the value
  clocks   nvidia-smi samples from the start of the warm-up to the end of the
           timed region
  cpu_baseline  the fp64 oracle timed on this host's cores on a bounded gate
           sample of the same workload

``--path banded-rerun`` times pa_run on a layout built before the timed region
instead (labelled as a re-run figure). ``--impl reference`` times the oracle
alone (rank 0), on the same workload and metric. ``--oracle-single`` times the
oracle on one host thread on configs 1..3.

``--partition density|fixed`` times the paper's (gate, window) thread partition
instead (one thread per gate window, a global atomic per event);
``--partition-sweep`` compares the event-density-aware partition (n_evt,tgt =
8; parallelism floors 1, 16 and 256) with globally fixed windows of 2 .. 32
cycles on one workload, one JSON line
per setting with the fused-kernel time and the thread statistics (thread
count, events per thread at the 50th/90th/99th percentile and the maximum), the
comparison of the paper's Figs. 19 and 20 (the large skewed workload,
``--config 3``, keeps the fixed settings' thread counts moderate), followed by
the library's own event-count partition (unbanded, then banded) on the same
workload.
Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..6] [--synth KNOB=VALUE ...]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "events/sec (dyn+leak) at 1 GB300; achieved HBM GB/s as % of roofline"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle sample time")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=["pass", "banded-rerun"], default="pass",
                    help="pass (default): every timed step is a whole pa_run on the loaded per-pin layout "
                         "(partition + fused kernel + final reduction); banded-rerun: pa_run on a cycle-banded "
                         "layout built before the timed region (a re-run figure)")
    ap.add_argument("--no-banded", action="store_true",
                    help="skip the banded layout's build / re-run figures and its e2e path")
    ap.add_argument("--warmup-seconds", type=float, default=1.0, help="minimum warm-up time")
    ap.add_argument("--oracle-single", action="store_true",
                    help="time the oracle on one host thread on configs 1..3 (bounded samples) and exit")
    ap.add_argument("--band-cycles", type=int, default=0, help="cycles per band (0 = library default)")
    ap.add_argument("--tile-events", type=int, default=0,
                    help="work partition knob: target events per light tile (0 = the library's default)")
    ap.add_argument("--heavy-events", type=int, default=0,
                    help="work partition knob: gates with more events are heavy (0 = the library's default); "
                         "tile + heavy above 448 selects the CTA kernel (k_fused) instead of the warp kernel")
    ap.add_argument("--partition", choices=["events", "density", "fixed"], default="events",
                    help="work partition: the library's event-count partition (default) or the paper's "
                         "(gate, window) threads, event-density-aware or globally fixed")
    ap.add_argument("--n-evt-tgt", type=int, default=8, help="density partition: target events per thread")
    ap.add_argument("--n-thr-floor", type=int, default=1, help="density partition: parallelism floor")
    ap.add_argument("--n-cyc-fix", type=int, default=8, help="fixed partition: cycles per thread")
    ap.add_argument("--partition-sweep", action="store_true",
                    help="time the density partition against fixed windows of 2..32 cycles (one line each)")
    ap.add_argument("--synth", nargs="*", default=[], metavar="KNOB=VALUE",
                    help="generator overrides for a scaled-down profiling case, e.g. n_gates=1000000 "
                         "n_events=200000000 (the line then names the workload as modified)")
    return ap.parse_args()


# ----------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Dist:
    def __init__(self, backend):
        self.world, self.rank, self.local = dist_env()
        self.pg = None
        if self.world > 1:
            import torch.distributed as td
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            td.init_process_group(backend)
            self.pg = td

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = torch.device("cuda", self.local) if torch.cuda.is_available() else torch.device("cpu")
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------- clocks

def gpu_local_cpus(dev: int):
    """CPUs of the GPU's own NUMA node (from sysfs, via its PCI address), as
    allowed for this process; None when they cannot be found. Pinned host
    buffers first touched from these CPUs live next to the GPU, so host <->
    device copies do not cross to the other socket."""
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(dev), "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip().lower()
        dom, rest = bus.split(":", 1)
        path = f"/sys/bus/pci/devices/{int(dom, 16):04x}:{rest}/local_cpulist"
        cpus = set()
        for part in open(path).read().strip().split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        return cpus or None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples (200 ms) while timed work runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        self.sel = self._selector(device_index)
        self.active = False
        self._t = None

    @staticmethod
    def _selector(idx):
        try:
            import torch
            u = str(torch.cuda.get_device_properties(idx).uuid)
            if u and not u.startswith("GPU-"):
                u = "GPU-" + u
            return ["-i", u]
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            first = vis.split(",")[idx] if vis else str(idx)
            return ["-i", first]

    def start(self):
        cmd = ["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            if self.active:
                self.rows.append(line.strip())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- workload

def pinned_alloc():
    import torch
    keep = []

    def alloc(shape, dtype):
        n = int(np.prod(shape))
        tt = torch.empty(n * np.dtype(dtype).itemsize, dtype=torch.uint8, pin_memory=True)
        keep.append(tt)
        return tt.numpy().view(dtype).reshape(shape)
    return alloc, keep


def algorithmic_bytes(w) -> int:
    """Bytes the method must move once per pass: events (t + slew, 8 B each),
    pin offsets (8 B per pin + 1), per-gate cell id, load and initial state
    (4 + 4 + 1 B), per-cycle outputs (waveform f32 + two u32 counts) and the
    tables."""
    return int(8 * w.n_events + 8 * (w.n_pins + 1) + 9 * w.n_gates + 12 * w.n_cycles
               + 4 * len(w.lut) + 4 * len(w.leak))


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gate_level_power_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    with open(os.path.join(ROOT, "include", "pa.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, config: int):
    """DRAM bytes per launch of `kernel` on `config` from a committed ncu
    summary under profiles/, if it was taken on the current kernel source
    (else None)."""
    pat = re.compile(r"traffic_bytes_per_launch\s+%s\s+config%d:\s*([0-9.eE+]+)\s+source:\s*([0-9a-f]+)"
                     % (re.escape(kernel), config))
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    for name in sorted(os.listdir(d)):
        if not name.endswith(".md"):
            continue
        m = pat.search(open(os.path.join(d, name)).read())
        if m and m.group(2) == kernel_source_digest():
            return float(m.group(1))
    return None


def cpu_baseline(config, seed, target_s, n_events_total, n_gates_total, **over):
    """Time the oracle (fp64, as it stands) on a contiguous gate block of the
    workload, grown until one run takes about target_s."""
    import oracle
    import synth
    cores = os.cpu_count() or 1
    g0 = n_gates_total // 3
    n = max(64, min(n_gates_total, 2000))
    el = 0.0
    while True:
        w = synth.generate_range(config, g0, min(n_gates_total, g0 + n), seed=seed, **over)
        t0 = time.perf_counter()
        oracle.run(w, threads=cores)
        el = time.perf_counter() - t0
        if el >= 0.5 * target_s or n >= n_gates_total or g0 + n >= n_gates_total:
            break
        grow = target_s / max(el, 1e-3)
        n = int(min(n_gates_total - g0, max(2 * n, n * min(grow, 50))))
    ev = w.n_events
    return {"value": ev / el, "unit": "events/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle, full waveform, gates [{g0}, {g0 + w.n_gates}) of {n_gates_total} "
                      f"({ev} of {n_events_total} events), {el:.2f} s on {cores} threads"}


# ----------------------------------------------------------------- reference arm

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    import synth
    over = synth_overrides(args.synth)
    cfg = synth.make_cfg(args.config, args.seed, **over)
    G, _, E = synth.sizes(args.config, args.seed, **over)
    cores = os.cpu_count() or 1
    # size the per-step sample so warmup + steps take a few minutes at most
    probe = synth.generate_range(args.config, G // 3, G // 3 + 2000, seed=args.seed, **over)
    t0 = time.perf_counter()
    oracle.run(probe, threads=cores)
    per_gate = (time.perf_counter() - t0) / probe.n_gates
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(200, min(G // 3, budget / max(per_gate, 1e-9))))
    w = synth.generate_range(args.config, G // 3, G // 3 + n, seed=args.seed, **over)
    for _ in range(args.warmup):
        oracle.run(w, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run(w, threads=cores)
    el = time.perf_counter() - t0
    v = w.n_events * args.steps / el
    sample = (f"fp64 oracle, full waveform, gates [{G // 3}, {G // 3 + w.n_gates}) of {G} "
              f"({w.n_events} of {E} events) per step, {cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "events/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args.config, G, E, cfg),
            "cpu_baseline": {"value": v, "unit": "events/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "events/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def synth_overrides(items):
    out = {}
    for it in items:
        k, v = it.split("=", 1)
        out[k] = float(v) if any(ch in v for ch in ".e") and not v.isdigit() else int(v)
    return out


def workload_config(config, G, E, cfg):
    import synth
    return {"workload": f"config {config}: " + synth.CONFIG_NAMES.get(config, "custom"),
            "gates": G, "events": E, "cycles": int(cfg.n_cycles), "t_clk_ns": float(cfg.t_clk_ns),
            "seed": int(cfg.seed),
            "l2": "inputs larger than L2 (events alone exceed 129 MB); no flush between steps"
            if E * 8 > 256e6 else "inputs smaller than L2: L2 not flushed (context only)"}


# ----------------------------------------------------------------- our arm

def run_ours(args):
    import torch

    import gate_level_power_gb300 as glp
    import synth
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = Dist("nccl")
    glp.load_library()
    alloc, keep = pinned_alloc()
    t0 = time.perf_counter()
    over = synth_overrides(args.synth)
    # the trace's pinned pages are first written by the generator: do that on the GPU's own socket
    all_cpus = os.sched_getaffinity(0)
    near = gpu_local_cpus(local)
    if near:
        os.sched_setaffinity(0, near)
    try:
        w = synth.generate(args.config, seed=args.seed, alloc=alloc, threads=len(near or all_cpus), **over)
    finally:
        os.sched_setaffinity(0, all_cpus)
    host_placement = (f"trace generated on the GPU-local CPUs ({len(near)} of {len(all_cpus)})" if near
                      else "GPU-local CPUs not found: default placement")
    gen_s = time.perf_counter() - t0
    cfg = synth.make_cfg(args.config, args.seed, **over)
    E, G, N = w.n_events, w.n_gates, w.n_cycles
    stream = torch.cuda.Stream(device=local)
    pa = glp.PowerAnalyzer(local, stream.cuda_stream)
    pa.load_workload(w)
    windows = args.partition != "events" or args.partition_sweep
    rerun = args.path == "banded-rerun" and not windows
    build_ms = None
    if rerun:  # a re-run figure: the layout is built before the timed region (reported as such)
        t0 = time.perf_counter()
        pa.build_bands(w.t_clk_ns, args.band_cycles)
        build_ms = (time.perf_counter() - t0) * 1e3
    wave = np.empty(N, np.float32)
    evc = np.empty(N, np.uint32)
    glc = np.empty(N, np.uint32)
    out = dict(waveform=wave, event_count=evc, glitch_count=glc)

    part = dict(partition=args.partition, n_evt_tgt=args.n_evt_tgt, n_thr_floor=args.n_thr_floor,
                n_cyc_fix=args.n_cyc_fix, tile_events=args.tile_events, heavy_events=args.heavy_events)

    def step(timing=False):
        return pa.run(w.vdd, w.t_clk_ns, N, out=out, timing=timing, **part)

    if args.partition_sweep:
        return partition_sweep(args, pa, w, out, dist, rank)

    # clocks are sampled from the start of the warm-up to the end of the
    # device-resident timed region
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    clk.active = True
    # warm-up: at least --warmup steps (3 at least) and at least --warmup-seconds
    t0 = time.perf_counter()
    n_warm = 0
    while n_warm < max(3, args.warmup) or time.perf_counter() - t0 < args.warmup_seconds:
        step()
        n_warm += 1
    warm_s = time.perf_counter() - t0
    # ---- device-resident timed region
    dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    fused_ms, pass_ms = [], []
    launches = 0
    for _ in range(args.steps):
        r = step(timing=True)
        fused_ms.append(r["ms_fused"])
        pass_ms.append(r["ms_total"])
        launches += r["kernel_launches"]
    e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    el_ms = e0.elapsed_time(e1)
    el_ms = dist.max(el_ms)
    value = world * E * args.steps / (el_ms * 1e-3)
    med_pass = dist.max(statistics.median(pass_ms))
    # a running nvidia-smi poller measurably slows host-to-device copies (some
    # 8 GB copies took 55-67 ms instead of 38 ms while it ran): stop it before
    # the end-to-end runs
    clk.active = False
    clk.stop()
    B = algorithmic_bytes(w)
    peak, peak_kind = hbm_peak()
    # ---- the cycle-banded layout beside the timed pass: its build, then runs
    # on it (the re-run figure of a trace analysed at several voltages or
    # window ends); reported, not the value
    banded = None
    if not windows and not rerun and not args.no_banded:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pa.build_bands(w.t_clk_ns, args.band_cycles)
        torch.cuda.synchronize()
        b_ms = (time.perf_counter() - t0) * 1e3
        for _ in range(3):
            step()
        rr = [step(timing=True) for _ in range(max(10, min(args.steps, 50)))]
        k_ms = statistics.median(x["ms_fused"] for x in rr)
        run_ms = statistics.median(x["ms_total"] for x in rr)
        banded = {"path": "banded" if rr[-1]["path"] == glp.PA_PATH_BANDED else "unbanded",
                  "build_ms": b_ms, "rerun_ms_median": run_ms, "k_band_ms_median": k_ms,
                  "rerun_events_per_s": E / (run_ms * 1e-3),
                  "build_plus_run_events_per_s": E / ((b_ms + run_ms) * 1e-3),
                  "rerun_roofline_frac": B / (k_ms * 1e-3) / 1e9 / peak,
                  "note": "pa_build_bands (layout build, once per trace and clock) then pa_run on the layout; "
                          "steps = " + str(len(rr))}
    # ---- end to end through the public API, host buffers
    h2d = 8 * (w.n_pins + 1) + 4 * E + 4 * E + E
    d2h = 4 * N + 4 * N + 4 * N + 4 * 8
    e2e_value = None
    e2e_paths = {}
    e2e_step_ms = {}
    if args.e2e_steps > 0:
        # A one-shot run through the public API: load the step's events from
        # pinned host memory and run, either straight on the loaded per-pin
        # layout (unbanded kernel) or after building the cycle-banded layout,
        # or stream the trace through the device. All are timed; the fastest
        # is the headline (a user running a trace once takes it), the others
        # are reported beside it.
        def e2e_step(path):
            if path == "stream_run":  # pa_run_stream: chunk copies overlapping the computation
                pa.run(w.vdd, w.t_clk_ns, N, out=out, stream=(w.pin_off, w.t_ns, w.slew_ps, w.value))
                return
            pa.load_events(w.pin_off, w.t_ns, w.slew_ps, w.value)
            if path == "load_build_bands_run":
                pa.build_bands(w.t_clk_ns, args.band_cycles)
            step()
        paths = (["load_run_windows"] if windows
                 else ["stream_run", "load_run_unbanded"] + ([] if args.no_banded else ["load_build_bands_run"]))
        for path in paths:
            for _ in range(2):
                e2e_step(path)
            dist.barrier()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            step_ms = []
            for _ in range(args.e2e_steps):
                ts = time.perf_counter()
                e2e_step(path)  # synchronous: returns once the results are on the host
                step_ms.append(round((time.perf_counter() - ts) * 1e3, 2))
            torch.cuda.synchronize()
            e2e_s = dist.max(time.perf_counter() - t0)
            e2e_paths[path] = world * E * args.e2e_steps / e2e_s
            e2e_step_ms[path] = step_ms
        e2e_value = max(e2e_paths.values())
        # the same bytes copied host -> device by a plain pinned-memory copy
        # (torch, no library code), the same number of times: the copies'
        # own step times, so that slow steps of the one-shot paths can be
        # told apart from slow steps of the host link
        dt = torch.empty(E, dtype=torch.float32, device=local)
        ds = torch.empty(E, dtype=torch.float32, device=local)
        dv = torch.empty(E, dtype=torch.uint8, device=local)
        ht, hs, hv = torch.from_numpy(w.t_ns), torch.from_numpy(w.slew_ps), torch.from_numpy(w.value)
        copy_ms = []
        for _ in range(args.e2e_steps + 2):
            torch.cuda.synchronize()
            ts = time.perf_counter()
            with torch.cuda.stream(stream):
                dt.copy_(ht, non_blocking=True)
                ds.copy_(hs, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
            stream.synchronize()
            copy_ms.append(round((time.perf_counter() - ts) * 1e3, 2))
        copy_ms = copy_ms[2:]
        del dt, ds, dv
    # ---- roofline of the fused kernel of the timed pass
    fused_mean = statistics.mean(fused_ms)
    fused_med = statistics.median(fused_ms)
    achieved = B / (fused_mean * 1e-3) / 1e9
    kname = {glp.PA_PATH_BANDED: "k_band", glp.PA_PATH_WINDOWS: "k_window", glp.PA_PATH_WARP: "k_csr"}.get(
        r["path"], "k_fused")
    traffic = None if args.synth else ncu_traffic(kname, args.config)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.config, args.seed, args.cpu_seconds, E, G, **over)
    if rank == 0:
        step_what = ("pa_run on a cycle-banded layout built before the timed region (re-run figure; the "
                     "layout build is not timed)" if rerun else
                     "pa_run on the loaded per-pin layout: the paper's partition (k_win_plan) + k_window + final "
                     "reduction" if windows else
                     "pa_run on the loaded per-pin layout: event-count partition (k_cp_*: light tiles and "
                     "heavy-gate pieces) + fused kernel (k_csr, one warp per item) + final reduction, every step"
                     if r["path"] == glp.PA_PATH_WARP else
                     "pa_run on the loaded per-pin layout: event-count partition (k_part_*) + fused kernel "
                     "(k_fused) + final reduction, every step")
        line = {
            "metric": METRIC, "value": value, "unit": "events/s", "n_gpus": world, "steps": args.steps,
            "warmup": n_warm, "ms_per_step": el_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(args.config, G, E, cfg),
                           **({"modified": " ".join(args.synth)} if args.synth else {})),
            "step": step_what,
            "ms_per_step_median": med_pass,
            "value_at_median_step": world * E / (med_pass * 1e-3),
            "warmup_seconds": warm_s,
            "gate_cycles_per_s": world * G * N * args.steps / (el_ms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": kname + " (fused dynamic + leakage power"
                         + (", with the unbanded kernel streaming big gates)" if r["path"] == glp.PA_PATH_BANDED
                            else ", the paper's (gate, window) threads)" if r["path"] == glp.PA_PATH_WINDOWS
                            else ")"),
                         "algorithmic_bytes_per_launch": B, "mean_launch_ms": fused_mean,
                         "median_launch_ms": fused_med,
                         "frac_at_median_launch": B / (fused_med * 1e-3) / 1e9 / peak,
                         "pass_frac": B / (statistics.mean(pass_ms) * 1e-3) / 1e9 / peak,
                         "peak_source": f"{peak_kind} HBM copy bandwidth"},
            "cpu_baseline": cpu,
            "banded_layout": banded,
            "e2e": None if e2e_value is None else {"value": e2e_value, "unit": "events/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": args.e2e_steps, "paths": e2e_paths,
                    "step_ms": e2e_step_ms,
                    "plain_copy_step_ms": copy_ms,
                    "plain_copy_note": "the steps' event bytes (times, slews, values) copied host -> device by a "
                                       "plain pinned-memory copy after the paths, for comparison",
                    "paths_at_median_step": {k: world * E / (statistics.median(v) * 1e-3)
                                             for k, v in e2e_step_ms.items() if v},
                    "note": "per step from pinned host memory: pa_run_stream (chunked copies overlapping "
                            "validation and the unbanded kernel), or pa_load_events (device-side validation) + "
                            "pa_run (+ pa_build_bands before it on the banded path); waveform/count copy to host; "
                            "library and netlist loaded once; value = the fastest path"},
            "clocks": clk.summary(),
            "gpu_launches": launches,
            "gen_seconds": gen_s,
            "host_placement": host_placement,
            "p_total_w": r["p_int"] + r["p_sw"] + r["p_gl"] + r["p_leak"],
            "n_tiles": r["n_tiles"], "n_heavy": r["n_heavy"],
            "path": {glp.PA_PATH_BANDED: "banded", glp.PA_PATH_WINDOWS: "windows",
                     glp.PA_PATH_WARP: "unbanded, warp kernel"}.get(r["path"], "unbanded"),
            **({"partition": dict(part, part_threads=r["part_threads"])} if windows else {}),
            **({"build_bands_ms": build_ms} if build_ms is not None else {}),
        }
        print(json.dumps(line), flush=True)
    pa.close()
    dist.close()
    del keep
    return 0


def oracle_single(args):
    """The oracle on one host thread, on a bounded gate sample of each of
    configs 1..3 (grown until one run takes about --cpu-seconds): one JSON
    line per configuration, events/s and gate-cycles/s of the sample."""
    import oracle
    import synth
    for config in (1, 2, 3):
        G, _, E = synth.sizes(config, args.seed)
        cfg = synth.make_cfg(config, args.seed)
        g0 = 0 if G <= 2000 else G // 3
        n = min(G, 2000)
        while True:
            w = synth.generate_range(config, g0, min(G, g0 + n), seed=args.seed)
            t0 = time.perf_counter()
            oracle.run(w, threads=1)
            el = time.perf_counter() - t0
            if el >= 0.5 * args.cpu_seconds or g0 + n >= G:
                break
            n = int(min(G - g0, max(2 * n, n * min(args.cpu_seconds / max(el, 1e-3), 50))))
        print(json.dumps({"metric": "oracle events/s, one host thread", "config": config,
                          "value": w.n_events / el, "unit": "events/s",
                          "gate_cycles_per_s": w.n_gates * int(cfg.n_cycles) / el, "threads": 1,
                          "sample": f"fp64 oracle, full waveform, gates [{g0}, {g0 + w.n_gates}) of {G} "
                                    f"({w.n_events} of {E} events), {el:.2f} s"}), flush=True)
    return 0


def partition_sweep(args, pa, w, out, dist, rank):
    """The paper's partition comparison (Figs. 19 and 20) on this GPU: the
    event-density-aware per-gate windows against globally fixed windows, on the
    same (gate, window) thread kernel. One JSON line per setting."""
    import torch
    settings = [dict(partition="density", n_evt_tgt=args.n_evt_tgt, n_thr_floor=f)
                for f in sorted({args.n_thr_floor, 16, 256})]
    settings += [dict(partition="fixed", n_cyc_fix=n) for n in (2, 4, 8, 16, 32)]
    # the library's own event-count partition beside them: event-count tiles of
    # the per-pin arrays (unbanded kernel), then the cycle-banded layout
    settings += [dict(partition="events"), dict(partition="events", banded=True)]
    steps = max(1, min(args.steps, 20))
    for st in settings:
        st = dict(st)
        if st.pop("banded", False):
            pa.build_bands(w.t_clk_ns, args.band_cycles)
        windows = st["partition"] != "events"
        s = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, out=out, part_stats=windows, **st)  # statistics, untimed
        for _ in range(max(3, args.warmup)):
            pa.run(w.vdd, w.t_clk_ns, w.n_cycles, out=out, **st)
        torch.cuda.synchronize()
        ms = [pa.run(w.vdd, w.t_clk_ns, w.n_cycles, out=out, timing=True, **st) for _ in range(steps)]
        fused = dist.max(statistics.median(m["ms_fused"] for m in ms))
        total = dist.max(statistics.median(m["ms_total"] for m in ms))
        if windows:
            work = {"threads": s["part_threads"],
                    "events_per_thread": dict(zip(("p50", "p90", "p99", "max"), s["part_evt"]))}
        else:
            work = {"path": {1: "banded", 3: "unbanded, warp kernel"}.get(s["path"], "unbanded"), "work_items": s["n_tiles"],
                    "heavy_items": s["n_heavy"]}
        if rank == 0:
            print(json.dumps({
                "metric": "fused kernel time, partition comparison", "unit": "ms", "value": fused,
                "ms_pass": total, "events_per_s": w.n_events / (total * 1e-3), "steps": steps,
                "config": {"workload": f"config {args.config}", "gates": w.n_gates, "events": w.n_events,
                           "cycles": w.n_cycles}, **st, **work,
            }), flush=True)
    pa.close()
    dist.close()
    return 0


def main():
    args = parse_args()
    if args.oracle_single:
        return oracle_single(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
