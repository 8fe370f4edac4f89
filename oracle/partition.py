"""Oracle of the paper's per-gate cycle partition (test infrastructure only).

Only ``tests/`` import this module. It
restates, in plain numpy and Python, the work decomposition of the
event-density-aware per-gate cycle partitioning of "GPU-Accelerated Gate-Level
Time-Based Power Analysis via Event-Density-Aware Partitioning and Kernel
Fusion" (Fig. 5; compared with a globally fixed partition in Figs. 19 and 20):
one thread per (gate g, window tau) of n_cyc^(g) cycles. It shares no code with
the CUDA library. The power results do not depend on the partition; what it
fixes is the thread count and the events each thread takes.

Readings taken where the extracted text lost its equations:

* density of gate g: rho = N_evt^(g) / N_cyc (events per cycle over the run);
* window of the parallelism floor: n_cyc,floor = ceil(N_cyc / N_thr,floor),
  and the density floor rho_floor = n_evt,tgt / n_cyc,floor;
* effective density rho_eff = rho + rho_floor (the additive form the text
  derives the thread count from);
* cycles per thread n_cyc^(g) = floor(n_evt,tgt / rho_eff + 1/2), clamped to
  [1, N_cyc] ("integer rounding": to nearest, halves up), every quantity in
  IEEE fp64 in that order of operations;
* globally fixed partition: n_cyc^(g) = min(n_cyc^fix, N_cyc) for every gate;
* thread tau of gate g holds cycles [tau n, min((tau + 1) n, N_cyc)), i.e. the
  time window [tau n T, min((tau + 1) n, N_cyc) T); threads per gate
  N_thr^(g) = ceil(N_cyc / n_cyc^(g)) (zero-event gates included);
* an event belongs to the window of its cycle c = floor(fl32(t / T)) (IEEE fp32
  division, as for the cycle bins), so window and bin membership agree;
* events-per-thread quantiles are nearest-rank: the q-th percentile of the n
  per-thread counts is the smallest x with at least ceil(q n / 100) counts
  <= x (0 when there are no threads).

Parity pins (tests/test_oracle_partition.py): a zero-event gate gets exactly
N_thr,floor threads when that divides N_cyc; a gate of density n_evt,tgt gets
one cycle per thread; the pages' additive approximation N_thr ~ N_evt /
n_evt,tgt + N_thr,floor holds in both limits; the fixed partition gives
ceil(N_cyc / n) threads per gate; per-thread counts from a brute-force walk
over every event, and their sum equals the event count.
"""
from __future__ import annotations

import math

import numpy as np

PART_DENSITY, PART_FIXED = 1, 2


def cycles_per_thread(n_evt_gate, n_cycles: int, mode: int, n_evt_tgt: int = 8, n_thr_floor: int = 1,
                      n_cyc_fix: int = 1) -> np.ndarray:
    """n_cyc^(g) for every gate (int64), from the per-gate event counts."""
    n_evt_gate = np.asarray(n_evt_gate, dtype=np.int64)
    N = int(n_cycles)
    if mode == PART_FIXED:
        return np.full(n_evt_gate.shape, max(1, min(int(n_cyc_fix), N)), dtype=np.int64)
    if mode != PART_DENSITY:
        raise ValueError("mode must be PART_DENSITY or PART_FIXED")
    n_floor = -(-N // int(n_thr_floor))                    # ceil(N_cyc / N_thr,floor)
    rho = n_evt_gate.astype(np.float64) / np.float64(N)    # events per cycle
    rho_floor = np.float64(n_evt_tgt) / np.float64(n_floor)
    x = np.float64(n_evt_tgt) / (rho + rho_floor)
    n = np.floor(x + np.float64(0.5)).astype(np.int64)
    return np.clip(n, 1, N)


def threads_per_gate(n_cyc_g, n_cycles: int) -> np.ndarray:
    """N_thr^(g) = ceil(N_cyc / n_cyc^(g))."""
    n_cyc_g = np.asarray(n_cyc_g, dtype=np.int64)
    return -(-int(n_cycles) // n_cyc_g)


def event_cycles(t_ns, t_clk_ns: float) -> np.ndarray:
    """Cycle of each event: floor(fl32(t / T)) with IEEE fp32 division."""
    q = np.asarray(t_ns, dtype=np.float32) / np.float32(t_clk_ns)
    return np.floor(q).astype(np.int64)


def gate_event_counts(w) -> np.ndarray:
    """N_evt^(g) of a workload (pins are gate-major: k inputs, then the output)."""
    pin_base = np.concatenate([[0], np.cumsum(w.n_inputs[w.cell_id].astype(np.int64) + 1)])
    po = np.asarray(w.pin_off, dtype=np.int64)
    return po[pin_base[1:]] - po[pin_base[:-1]]


def thread_event_counts(w, mode: int, n_evt_tgt: int = 8, n_thr_floor: int = 1, n_cyc_fix: int = 1) -> np.ndarray:
    """Events of every (gate, window) thread, gate-major then window order (int64)."""
    n_evt = gate_event_counts(w)
    n = cycles_per_thread(n_evt, w.n_cycles, mode, n_evt_tgt, n_thr_floor, n_cyc_fix)
    nthr = threads_per_gate(n, w.n_cycles)
    first = np.concatenate([[0], np.cumsum(nthr)])
    counts = np.zeros(int(first[-1]), dtype=np.int64)
    pin_base = np.concatenate([[0], np.cumsum(w.n_inputs[w.cell_id].astype(np.int64) + 1)])
    po = np.asarray(w.pin_off, dtype=np.int64)
    cyc = event_cycles(w.t_ns, w.t_clk_ns)
    gate_of_event = np.repeat(np.arange(len(n_evt), dtype=np.int64), n_evt)
    tau = cyc // n[gate_of_event]
    np.add.at(counts, first[gate_of_event] + tau, 1)
    return counts


def thread_event_counts_brute(w, mode: int, n_evt_tgt: int = 8, n_thr_floor: int = 1,
                              n_cyc_fix: int = 1) -> np.ndarray:
    """The same counts by a plain walk over gates, windows and events (tiny cases)."""
    n_evt = gate_event_counts(w)
    n = cycles_per_thread(n_evt, w.n_cycles, mode, n_evt_tgt, n_thr_floor, n_cyc_fix)
    T = np.float32(w.t_clk_ns)
    out = []
    e = 0
    for g in range(len(n_evt)):
        ng = int(n[g])
        windows = []
        c0 = 0
        while c0 < w.n_cycles:
            windows.append((c0, min(c0 + ng, int(w.n_cycles))))
            c0 += ng
        cnt = [0] * len(windows)
        for _ in range(int(n_evt[g])):
            c = int(math.floor(float(np.float32(w.t_ns[e]) / T)))
            for i, (a, b) in enumerate(windows):
                if a <= c < b:
                    cnt[i] += 1
            e += 1
        out.extend(cnt)
    return np.asarray(out, dtype=np.int64)


def nearest_rank(counts, q: int) -> int:
    """Smallest x with at least ceil(q n / 100) of the counts <= x (q in 1..100)."""
    c = np.sort(np.asarray(counts, dtype=np.int64))
    if len(c) == 0:
        return 0
    r = (q * len(c) + 99) // 100
    return int(c[max(r, 1) - 1])


def stats(w, mode: int, n_evt_tgt: int = 8, n_thr_floor: int = 1, n_cyc_fix: int = 1) -> dict:
    """Thread count and events-per-thread quantiles (p50, p90, p99, max)."""
    cnt = thread_event_counts(w, mode, n_evt_tgt, n_thr_floor, n_cyc_fix)
    return {"threads": int(len(cnt)), "p50": nearest_rank(cnt, 50), "p90": nearest_rank(cnt, 90),
            "p99": nearest_rank(cnt, 99), "max": int(cnt.max()) if len(cnt) else 0}
