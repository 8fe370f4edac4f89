"""Seeded synthetic workloads for gate-level time-based power analysis.

This package only draws inputs (library, netlist, per-pin event streams); it
holds none of the power arithmetic. The fp64 oracle and the CUDA path both
consume what it returns. The native generator (``synth.cpp``) is built by
``build()`` and loaded through ctypes.

Standard workloads (``config`` 1..5) follow the evaluation scale of "GPU-
Accelerated Gate-Level Time-Based Power Analysis via Event-Density-Aware
Partitioning and Kernel Fusion" (Section 5, Tables 2-5): gate counts, cell
mix, LUT sizes, cycle counts, event totals, activity skew, glitch share and
bursts. The paper's real designs and activity files are not available; these
seeded inputs stand in for them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cpp")
_LIB = os.path.join(_HERE, "libsynth.so")


class SynthCfg(ctypes.Structure):
    _fields_ = [
        ("config", ctypes.c_int32),
        ("seed", ctypes.c_uint64),
        ("n_gates", ctypes.c_int64),
        ("n_cells", ctypes.c_int32),
        ("k_mode", ctypes.c_int32),
        ("n_slew", ctypes.c_int32),
        ("n_load", ctypes.c_int32),
        ("n_cycles", ctypes.c_int32),
        ("t_clk_ns", ctypes.c_float),
        ("n_events", ctypes.c_int64),
        ("activity", ctypes.c_int32),
        ("zipf_s", ctypes.c_double),
        ("zipf_q", ctypes.c_double),
        ("top1_share", ctypes.c_double),
        ("slew_dist", ctypes.c_int32),
        ("load_dist", ctypes.c_int32),
        ("pair_frac", ctypes.c_double),
        ("pair_cycle_frac", ctypes.c_double),
        ("pair_w_lo_ns", ctypes.c_double),
        ("pair_w_hi_ns", ctypes.c_double),
        ("burst_frac", ctypes.c_double),
        ("burst_width", ctypes.c_int32),
        ("burst_cover", ctypes.c_double),
        ("quantum_ns", ctypes.c_double),
        ("vdd", ctypes.c_double),
        ("threads", ctypes.c_int32),
        ("toggles", ctypes.c_int32),
    ]


class SynthStats(ctypes.Structure):
    _fields_ = [
        ("n_pins", ctypes.c_uint64),
        ("n_events", ctypes.c_uint64),
        ("max_gate_events", ctypes.c_uint64),
        ("max_pin_events", ctypes.c_uint64),
        ("top1_share", ctypes.c_double),
        ("zipf_q", ctypes.c_double),
        ("glitch_events", ctypes.c_uint64),
        ("max_pin_cycle_events", ctypes.c_uint64),
        ("heavy_events_over_2048", ctypes.c_uint64),
    ]


CONFIG_NAMES = {
    1: "tiny: 1k gates, 4 cells (INV/NAND2/NOR2/XOR2), 7x7 LUTs, 100 cycles @ 1 ns, 10k events",
    2: "mid: 100k gates, 32 cells k=1..4, 7x7 LUTs, 1k cycles @ 1 ns, 10M events, glitch pulses in ~5% of cycles",
    3: "large skewed: 1M gates, 32 cells, 10k cycles @ 0.8 ns, 200M events, Zipf(1.2) top1%~50%, 15% glitch edges",
    4: "very large skewed: 5M gates, 64 cells k=1..4, 8x8 LUTs, 100k cycles @ 1 ns, 1B events, Zipf(1.1), lognormal slews",
    5: "bursty: 10M gates, 64 cells k=4, 8x8 LUTs, 50k cycles @ 1 ns, 2B events, 80% in 5% of cycles, Zipf(1.3)",
    6: "waveform-bin stress: 1k gates, 32 cells k=1..4, 100k cycles @ 1 ns, every pin toggling 4 times per cycle "
       "(knob toggles = 1, 2, 4, 8)",
}


def build(force: bool = False) -> str:
    """Compile the generator into ``libsynth.so`` next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp = ctypes.c_void_p
        L.synth_default.argtypes = [ctypes.POINTER(SynthCfg), ctypes.c_int32]
        L.synth_create.argtypes = [ctypes.POINTER(SynthCfg)]
        L.synth_create.restype = vp
        L.synth_destroy.argtypes = [vp]
        L.synth_get_cfg.argtypes = [vp, ctypes.POINTER(SynthCfg)]
        u64p = ctypes.POINTER(ctypes.c_uint64)
        L.synth_sizes.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), u64p, u64p, u64p, u64p, u64p]
        L.synth_fill_library.argtypes = [vp] + [vp] * 9
        L.synth_fill_netlist.argtypes = [vp] * 5
        L.synth_fill_events.argtypes = [vp] * 5 + [ctypes.POINTER(SynthStats)]
        L.synth_get_stats.argtypes = [vp, ctypes.POINTER(SynthStats)]
        L.synth_range.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, u64p, u64p, u64p, u64p]
        L.synth_fill_range.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp, vp, vp, vp]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


@dataclass
class Workload:
    """One generated workload: library, netlist, events and run parameters.

    Library arrays: ``n_inputs, n_slew, n_load`` (u8 [n_cells]), ``slew_axis,
    load_axis`` (f32 [n_cells, 8]), ``lut_off`` (u32), ``lut`` (f32, fJ, per cell
    ``[2^k][n_slew][n_load]``), ``leak_off`` (u32), ``leak`` (f32, nW, per cell
    ``[2^k]``). Netlist: ``cell_id`` (u32), ``load_ff`` (f32), ``init_in``,
    ``init_out`` (u8). Events: ``pin_off`` (u64 [P+1]), ``t_ns``, ``slew_ps``
    (f32 [E]), ``value`` (u8 [E]). Gate g owns pins ``pin_base[g] ..
    pin_base[g] + k``, inputs first, output last.
    """
    config: int
    seed: int
    vdd: float
    t_clk_ns: float
    n_cycles: int
    n_inputs: np.ndarray
    n_slew: np.ndarray
    n_load: np.ndarray
    slew_axis: np.ndarray
    load_axis: np.ndarray
    lut_off: np.ndarray
    lut: np.ndarray
    leak_off: np.ndarray
    leak: np.ndarray
    cell_id: np.ndarray
    load_ff: np.ndarray
    init_in: np.ndarray
    init_out: np.ndarray
    pin_off: np.ndarray
    t_ns: np.ndarray
    slew_ps: np.ndarray
    value: np.ndarray
    stats: dict = field(default_factory=dict)

    @property
    def n_gates(self) -> int:
        return int(self.cell_id.shape[0])

    @property
    def n_events(self) -> int:
        return int(self.t_ns.shape[0])

    @property
    def n_pins(self) -> int:
        return int(self.pin_off.shape[0] - 1)

    def pin_base(self) -> np.ndarray:
        k = self.n_inputs[self.cell_id].astype(np.uint64) + 1
        pb = np.zeros(self.n_gates + 1, dtype=np.uint64)
        np.cumsum(k, out=pb[1:])
        return pb


def make_cfg(config: int, seed: int = 0, **overrides) -> SynthCfg:
    L = _load()
    c = SynthCfg()
    L.synth_default(ctypes.byref(c), int(config))
    c.seed = int(seed)
    for k, v in overrides.items():
        if not hasattr(c, k):
            raise KeyError(f"unknown synth knob {k!r}")
        setattr(c, k, v)
    return c


def sizes(config: int, seed: int = 0, **overrides):
    """(gates, pins, events) of a workload, without drawing its events."""
    L = _load()
    cfg = make_cfg(config, seed, **overrides)
    h = L.synth_create(ctypes.byref(cfg))
    try:
        nc = ctypes.c_uint32()
        lut_len, leak_len, G, P, E = (ctypes.c_uint64() for _ in range(5))
        L.synth_sizes(h, ctypes.byref(nc), ctypes.byref(lut_len), ctypes.byref(leak_len),
                      ctypes.byref(G), ctypes.byref(P), ctypes.byref(E))
        return G.value, P.value, E.value
    finally:
        L.synth_destroy(h)


def generate(config: int, seed: int = 0, alloc=None, with_value: bool = True, **overrides) -> Workload:
    """Generate a workload. ``alloc(shape, dtype) -> ndarray`` may supply the
    large event arrays (e.g. views of pinned host memory)."""
    L = _load()
    cfg = make_cfg(config, seed, **overrides)
    h = L.synth_create(ctypes.byref(cfg))
    try:
        L.synth_get_cfg(h, ctypes.byref(cfg))
        nc = ctypes.c_uint32()
        lut_len, leak_len, G, P, E = (ctypes.c_uint64() for _ in range(5))
        L.synth_sizes(h, ctypes.byref(nc), ctypes.byref(lut_len), ctypes.byref(leak_len),
                      ctypes.byref(G), ctypes.byref(P), ctypes.byref(E))
        nc, G, P, E = nc.value, G.value, P.value, E.value
        A = alloc or (lambda shape, dtype: np.empty(shape, dtype=dtype))
        k = np.empty(nc, np.uint8); ns = np.empty(nc, np.uint8); nl = np.empty(nc, np.uint8)
        sax = np.empty((nc, 8), np.float32); lax = np.empty((nc, 8), np.float32)
        lut_off = np.empty(nc, np.uint32); leak_off = np.empty(nc, np.uint32)
        lut = np.empty(lut_len.value, np.float32); leak = np.empty(leak_len.value, np.float32)
        L.synth_fill_library(h, *(_ptr(a) for a in (k, ns, nl, sax, lax, lut_off, lut, leak_off, leak)))
        cell = np.empty(G, np.uint32); load = np.empty(G, np.float32)
        ii = np.empty(G, np.uint8); io = np.empty(G, np.uint8)
        L.synth_fill_netlist(h, _ptr(cell), _ptr(load), _ptr(ii), _ptr(io))
        pin_off = np.empty(P + 1, np.uint64)
        t = A((E,), np.float32)
        s = A((E,), np.float32)
        v = A((E,), np.uint8) if with_value else None
        st = SynthStats()
        L.synth_fill_events(h, _ptr(pin_off), _ptr(t), _ptr(s), _ptr(v) if v is not None else None,
                            ctypes.byref(st))
        stats = {name: getattr(st, name) for name, _ in SynthStats._fields_}
        return Workload(config=config, seed=seed, vdd=cfg.vdd, t_clk_ns=float(np.float32(cfg.t_clk_ns)),
                        n_cycles=cfg.n_cycles, n_inputs=k, n_slew=ns, n_load=nl, slew_axis=sax,
                        load_axis=lax, lut_off=lut_off, lut=lut, leak_off=leak_off, leak=leak,
                        cell_id=cell, load_ff=load, init_in=ii, init_out=io, pin_off=pin_off,
                        t_ns=t, slew_ps=s, value=v, stats=stats)
    finally:
        L.synth_destroy(h)


def generate_range(config: int, g0: int, g1: int, seed: int = 0, **overrides) -> Workload:
    """Gates [g0, g1) of a workload as a workload of their own (pin offsets
    rebased), identical to that slice of ``generate(config, seed)``. Lets a
    CPU sample of a large workload be drawn without generating all of it."""
    L = _load()
    cfg = make_cfg(config, seed, **overrides)
    h = L.synth_create(ctypes.byref(cfg))
    try:
        L.synth_get_cfg(h, ctypes.byref(cfg))
        nc = ctypes.c_uint32()
        lut_len, leak_len, G, P, E = (ctypes.c_uint64() for _ in range(5))
        L.synth_sizes(h, ctypes.byref(nc), ctypes.byref(lut_len), ctypes.byref(leak_len),
                      ctypes.byref(G), ctypes.byref(P), ctypes.byref(E))
        nc, G = nc.value, G.value
        g0, g1 = max(0, int(g0)), min(G, int(g1))
        k = np.empty(nc, np.uint8); ns = np.empty(nc, np.uint8); nl = np.empty(nc, np.uint8)
        sax = np.empty((nc, 8), np.float32); lax = np.empty((nc, 8), np.float32)
        lut_off = np.empty(nc, np.uint32); leak_off = np.empty(nc, np.uint32)
        lut = np.empty(lut_len.value, np.float32); leak = np.empty(leak_len.value, np.float32)
        L.synth_fill_library(h, *(_ptr(a) for a in (k, ns, nl, sax, lax, lut_off, lut, leak_off, leak)))
        cell = np.empty(G, np.uint32); load = np.empty(G, np.float32)
        ii = np.empty(G, np.uint8); io = np.empty(G, np.uint8)
        L.synth_fill_netlist(h, _ptr(cell), _ptr(load), _ptr(ii), _ptr(io))
        plo, phi, elo, ehi = (ctypes.c_uint64() for _ in range(4))
        L.synth_range(h, g0, g1, ctypes.byref(plo), ctypes.byref(phi), ctypes.byref(elo), ctypes.byref(ehi))
        n_p, n_e = phi.value - plo.value, ehi.value - elo.value
        pin_off = np.empty(n_p + 1, np.uint64)
        t = np.empty(n_e, np.float32); s = np.empty(n_e, np.float32); v = np.empty(n_e, np.uint8)
        L.synth_fill_range(h, g0, g1, _ptr(pin_off), _ptr(t), _ptr(s), _ptr(v))
        return Workload(config=config, seed=seed, vdd=cfg.vdd, t_clk_ns=float(np.float32(cfg.t_clk_ns)),
                        n_cycles=cfg.n_cycles, n_inputs=k, n_slew=ns, n_load=nl, slew_axis=sax,
                        load_axis=lax, lut_off=lut_off, lut=lut, leak_off=leak_off, leak=leak,
                        cell_id=cell[g0:g1].copy(), load_ff=load[g0:g1].copy(), init_in=ii[g0:g1].copy(),
                        init_out=io[g0:g1].copy(), pin_off=pin_off, t_ns=t, slew_ps=s, value=v,
                        stats={"gate_range": (g0, g1), "n_gates_total": G})
    finally:
        L.synth_destroy(h)


def custom(**kw) -> Workload:
    """A custom workload (config 0) with explicit knobs, for tests."""
    seed = kw.pop("seed", 0)
    return generate(0, seed=seed, **kw)
