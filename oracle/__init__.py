"""fp64 CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg import this package. It wraps ``oracle.c`` (plain C, fp64, serial per
gate), which follows Sections 2.4.1-2.4.2 and Fig. 7 of "GPU-Accelerated
Gate-Level Time-Based Power Analysis via Event-Density-Aware Partitioning and
Kernel Fusion"; see the header of ``oracle.c`` for the readings taken where the
extracted text is silent or lost its equations. It shares no code with the CUDA
library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

WAVE_FULL, WAVE_NONE, WAVE_SAMPLE = 0, 1, 2

_vp = ctypes.c_void_p


class OrLib(ctypes.Structure):
    _fields_ = [("n_cells", ctypes.c_uint32), ("k", _vp), ("ns", _vp), ("nl", _vp), ("sax", _vp),
                ("lax", _vp), ("lut_off", _vp), ("lut", _vp), ("leak_off", _vp), ("leak", _vp)]


class OrNet(ctypes.Structure):
    _fields_ = [("n_gates", ctypes.c_uint64), ("cell", _vp), ("load", _vp), ("init_in", _vp),
                ("init_out", _vp)]


class OrEv(ctypes.Structure):
    _fields_ = [("n_pins", ctypes.c_uint64), ("pin_off", _vp), ("t", _vp), ("slew", _vp), ("value", _vp)]


class OrPar(ctypes.Structure):
    _fields_ = [("vdd", ctypes.c_double), ("t_clk", ctypes.c_float), ("n_cycles", ctypes.c_uint32),
                ("t_max", ctypes.c_double), ("wave_mode", ctypes.c_int32), ("sample_cycles", _vp),
                ("n_sample", ctypes.c_uint32), ("gate_begin", ctypes.c_uint64),
                ("gate_end", ctypes.c_uint64), ("threads", ctypes.c_int32), ("glitch_mode", ctypes.c_int32),
                ("esw_mode", ctypes.c_int32)]


class OrOut(ctypes.Structure):
    _fields_ = [("e_int", ctypes.c_double), ("e_sw", ctypes.c_double), ("e_gl", ctypes.c_double),
                ("e_leak", ctypes.c_double), ("p_int", ctypes.c_double), ("p_sw", ctypes.c_double),
                ("p_gl", ctypes.c_double), ("p_leak", ctypes.c_double), ("t_max", ctypes.c_double),
                ("wave_energy", _vp), ("waveform", _vp), ("evcount", _vp), ("glcount", _vp),
                ("state_pre", _vp), ("lut_ij", _vp), ("is_glitch", _vp), ("gate_power", _vp)]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (plain C, no fast-math, no FMA contraction)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.or_run.argtypes = [ctypes.POINTER(OrLib), ctypes.POINTER(OrNet), ctypes.POINTER(OrEv),
                             ctypes.POINTER(OrPar), ctypes.POINTER(OrOut)]
        L.or_run.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def run(w, *, vdd=None, t_clk=None, n_cycles=None, t_max=0.0, wave="full", sample_cycles=None,
        gate_range=None, threads=1, debug=False, use_value=True, gate_power=False, glitch_mode=0,
        esw_mode=0):
    """Run the oracle on workload-like object ``w`` (attributes as in ``synth.Workload``).

    Returns a dict: ``p_int, p_sw, p_gl, p_leak`` (W), ``e_*`` (fJ), ``t_max``
    (ns), and, as requested, ``waveform`` (W per cycle, or per sampled cycle),
    ``wave_energy`` (fJ), ``evcount``/``glcount`` (u64 per cycle), and per-event
    debug arrays ``state_pre``, ``lut_ij``, ``is_glitch`` (filled only for the
    gates walked), and with ``gate_power`` the per-gate power ``gate_power``
    (W, [gates walked, 4]: internal, switching, glitch, leakage).
    """
    L = _load()
    vdd = w.vdd if vdd is None else vdd
    t_clk = w.t_clk_ns if t_clk is None else t_clk
    n_cycles = w.n_cycles if n_cycles is None else n_cycles
    keep = []

    def k(a, dt):
        a = _c(a, dt)
        keep.append(a)
        return _p(a)

    lib = OrLib(len(w.n_inputs), k(w.n_inputs, np.uint8), k(w.n_slew, np.uint8), k(w.n_load, np.uint8),
                k(w.slew_axis, np.float32), k(w.load_axis, np.float32), k(w.lut_off, np.uint32),
                k(w.lut, np.float32), k(w.leak_off, np.uint32), k(w.leak, np.float32))
    G = len(w.cell_id)
    net = OrNet(G, k(w.cell_id, np.uint32), k(w.load_ff, np.float32), k(w.init_in, np.uint8),
                k(w.init_out, np.uint8))
    value = w.value if use_value else None
    ev = OrEv(len(w.pin_off) - 1, k(w.pin_off, np.uint64), k(w.t_ns, np.float32), k(w.slew_ps, np.float32),
              k(value, np.uint8) if value is not None else None)
    g0, g1 = (0, G) if gate_range is None else gate_range
    mode = {"full": WAVE_FULL, "none": WAVE_NONE, "sample": WAVE_SAMPLE}[wave]
    sc = None
    if mode == WAVE_SAMPLE:
        sc = np.ascontiguousarray(sample_cycles, dtype=np.uint32)
        keep.append(sc)
    par = OrPar(float(vdd), float(t_clk), int(n_cycles), float(t_max), mode, _p(sc),
                0 if sc is None else len(sc), int(g0), int(g1), int(threads), int(glitch_mode), int(esw_mode))
    out = OrOut()
    res = {}
    nb = n_cycles if mode == WAVE_FULL else (len(sc) if mode == WAVE_SAMPLE else 0)
    if nb:
        res["wave_energy"] = np.zeros(nb, np.float64)
        res["waveform"] = np.zeros(nb, np.float64)
        out.wave_energy = _p(res["wave_energy"])
        out.waveform = _p(res["waveform"])
    res["evcount"] = np.zeros(n_cycles, np.uint64)
    res["glcount"] = np.zeros(n_cycles, np.uint64)
    out.evcount = _p(res["evcount"])
    out.glcount = _p(res["glcount"])
    if debug:
        E = len(w.t_ns)
        for name in ("state_pre", "lut_ij", "is_glitch"):
            res[name] = np.full(E, 0xEE, np.uint8)
            setattr(out, name, _p(res[name]))
    if gate_power:
        res["gate_power"] = np.zeros((g1 - g0, 4), np.float64)
        out.gate_power = _p(res["gate_power"])
    rc = L.or_run(ctypes.byref(lib), ctypes.byref(net), ctypes.byref(ev), ctypes.byref(par), ctypes.byref(out))
    if rc != 0:
        raise RuntimeError(f"oracle failed (rc={rc})")
    for name in ("e_int", "e_sw", "e_gl", "e_leak", "p_int", "p_sw", "p_gl", "p_leak", "t_max"):
        res[name] = getattr(out, name)
    return res
