"""Helpers for tests: hand-made workloads and an independent brute-force
formulation of the power computation (used to pin the oracle)."""
import json
import math
import os
from types import SimpleNamespace

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def workload(library, netlist, events, params):
    lib, net, ev = library, netlist, events
    w = SimpleNamespace(
        config=0, seed=0,
        vdd=float(params["vdd"]), t_clk_ns=float(np.float32(params["t_clk_ns"])),
        n_cycles=int(params["n_cycles"]),
        n_inputs=np.asarray(lib["n_inputs"], np.uint8), n_slew=np.asarray(lib["n_slew"], np.uint8),
        n_load=np.asarray(lib["n_load"], np.uint8),
        slew_axis=np.asarray(lib["slew_axis"], np.float32).reshape(-1, 8),
        load_axis=np.asarray(lib["load_axis"], np.float32).reshape(-1, 8),
        lut_off=np.asarray(lib["lut_off"], np.uint32), lut=np.asarray(lib["lut"], np.float32),
        leak_off=np.asarray(lib["leak_off"], np.uint32), leak=np.asarray(lib["leak"], np.float32),
        cell_id=np.asarray(net["cell_id"], np.uint32), load_ff=np.asarray(net["load_ff"], np.float32),
        init_in=np.asarray(net["init_in"], np.uint8), init_out=np.asarray(net["init_out"], np.uint8),
        pin_off=np.asarray(ev["pin_off"], np.uint64), t_ns=np.asarray(ev["t_ns"], np.float32),
        slew_ps=np.asarray(ev["slew_ps"], np.float32),
        value=None if ev.get("value") is None else np.asarray(ev["value"], np.uint8),
        stats={})
    w.t_max_ns = float(params.get("t_max_ns", 0.0))
    return w


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        d = json.load(f)
    return workload(d["library"], d["netlist"], d["events"], d["params"]), d


def pin_base(w):
    k = w.n_inputs[w.cell_id].astype(np.int64) + 1
    pb = np.zeros(len(w.cell_id) + 1, np.int64)
    np.cumsum(k, out=pb[1:])
    return pb


def values_of(w):
    """New value per event: the given array, else toggles from the initial pin values."""
    if w.value is not None:
        return w.value.astype(np.int64)
    pb = pin_base(w)
    v = np.zeros(len(w.t_ns), np.int64)
    for g in range(len(w.cell_id)):
        k = int(w.n_inputs[w.cell_id[g]])
        for q in range(k + 1):
            a, b = int(w.pin_off[pb[g] + q]), int(w.pin_off[pb[g] + q + 1])
            init = (int(w.init_in[g]) >> q) & 1 if q < k else int(w.init_out[g])
            for i in range(a, b):
                v[i] = init ^ ((i - a + 1) & 1)
    return v


def brute_force(w, vdd=None, t_clk=None, n_cycles=None, t_max=0.0, glitch_mode=0, esw_mode=0):
    """A second, structurally different fp64 formulation for tiny workloads.

    Instead of a k-way merge it evaluates the gate state as a function of time
    ("value of the last event at or before tau" per input pin), integrates
    leakage piecewise over the union of event times and cycle boundaries, and
    classifies each event by counting the earlier events of its pin in its
    cycle. O(E^2); for a handful of gates only. glitch_mode 1: every event of
    a pin-cycle with two or more events is a glitch (the first takes the pulse
    to the next event); esw_mode 1: C V^2 per rising output edge only.
    """
    vdd = w.vdd if vdd is None else vdd
    Tf = np.float32(w.t_clk_ns if t_clk is None else t_clk)
    T = float(Tf)
    n_cyc = w.n_cycles if n_cycles is None else n_cycles
    tm = t_max if t_max > 0 else n_cyc * T
    vals = values_of(w)
    pb = pin_base(w)
    E = len(w.t_ns)
    out = dict(e_int=0.0, e_sw=0.0, e_gl=0.0, e_leak=0.0,
               wave_energy=np.zeros(n_cyc), evcount=np.zeros(n_cyc, np.int64),
               glcount=np.zeros(n_cyc, np.int64), state_pre=np.zeros(E, np.int64),
               lut_ij=np.zeros(E, np.int64), is_glitch=np.zeros(E, np.int64),
               gate_energy=np.zeros((len(w.cell_id), 4)))
    for g in range(len(w.cell_id)):
        tot0 = [out["e_int"], out["e_sw"], out["e_gl"], out["e_leak"]]
        cell = int(w.cell_id[g]); k = int(w.n_inputs[cell])
        ns, nl = int(w.n_slew[cell]), int(w.n_load[cell])
        sax = [float(x) for x in w.slew_axis[cell][:ns]]; lax = [float(x) for x in w.load_axis[cell][:nl]]
        C = float(w.load_ff[g])
        pins = []
        for q in range(k + 1):
            a, b = int(w.pin_off[pb[g] + q]), int(w.pin_off[pb[g] + q + 1])
            pins.append([(float(w.t_ns[i]), float(w.slew_ps[i]), int(vals[i]), i) for i in range(a, b)])
        init = [(int(w.init_in[g]) >> q) & 1 for q in range(k)]

        def state(tau, inclusive):
            S = 0
            for q in range(k):
                v = init[q]
                for (t, _, val, _) in pins[q]:
                    if t < tau or (inclusive and t == tau):
                        v = val
                S |= v << q
            return S

        def table(S, i, j):
            return float(w.lut[int(w.lut_off[cell]) + (S * ns + i) * nl + j])

        # dynamic energy per event
        for q in range(k + 1):
            for n, (t, s, val, idx) in enumerate(pins[q]):
                c = int(math.floor(np.float32(t) / Tf))
                S = state(t, inclusive=False)
                same_cycle = [m for m, (t2, *_r) in enumerate(pins[q])
                              if int(math.floor(np.float32(t2) / Tf)) == c]
                earlier_same_cycle = sum(1 for m in same_cycle if m < n)
                glitch = earlier_same_cycle >= 1 or (glitch_mode == 1 and len(same_cycle) >= 2)
                out["evcount"][c] += 1
                if q < k:
                    i = max([m for m in range(ns - 1) if sax[m] <= s] + [0])
                    j = max([m for m in range(nl - 1) if lax[m] <= C] + [0])
                    u = (s - sax[i]) / (sax[i + 1] - sax[i]); v = (C - lax[j]) / (lax[j + 1] - lax[j])
                    e_int = (table(S, i, j) * (1 - u) * (1 - v) + table(S, i + 1, j) * u * (1 - v)
                             + table(S, i, j + 1) * (1 - u) * v + table(S, i + 1, j + 1) * u * v)
                    e_sw = 0.0
                    out["lut_ij"][idx] = (i << 4) | j
                else:
                    e_int = 0.0
                    e_sw = 0.5 * C * vdd * vdd if esw_mode == 0 else (C * vdd * vdd if val == 1 else 0.0)
                    out["lut_ij"][idx] = 0xFF
                out["state_pre"][idx] = S
                out["is_glitch"][idx] = int(glitch)
                if glitch:
                    if earlier_same_cycle >= 1:
                        tp, sp = pins[q][n - 1][0], pins[q][n - 1][1]
                        pw = t - tp
                    else:  # the first edge of the cycle: the pulse to the next event
                        tp, sp = pins[q][n + 1][0], pins[q][n + 1][1]
                        pw = tp - t
                    r = min(1.0, pw * 1000.0 / ((s + sp) / 2.0))
                    out["e_gl"] += r * (e_int + e_sw)
                    out["wave_energy"][c] += r * (e_int + e_sw)
                    out["glcount"][c] += 1
                else:
                    out["e_int"] += e_int; out["e_sw"] += e_sw
                    out["wave_energy"][c] += e_int + e_sw
        # leakage: piecewise over event times and cycle boundaries
        cuts = {0.0, tm} | {c * T for c in range(n_cyc + 1) if c * T < tm}
        for q in range(k):
            cuts |= {t for (t, *_r) in pins[q] if t < tm}
        cuts = sorted(cuts)
        for a, b in zip(cuts[:-1], cuts[1:]):
            p = float(w.leak[int(w.leak_off[cell]) + state(a, inclusive=True)])
            e = p * (b - a) * 1e-3
            out["e_leak"] += e
            c = int(math.floor(0.5 * (a + b) / T))
            if c < n_cyc:
                out["wave_energy"][c] += e
        # this gate's share of each total
        for m, name in enumerate(("e_int", "e_sw", "e_gl", "e_leak")):
            out["gate_energy"][g, m] = out[name] - tot0[m]
    out["gate_power"] = out["gate_energy"] / tm * 1e-6
    for name in ("int", "sw", "gl", "leak"):
        out["p_" + name] = out["e_" + name] / tm * 1e-6
    out["waveform"] = out["wave_energy"] / T * 1e-6
    out["t_max"] = tm
    return out
