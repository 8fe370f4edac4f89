"""Gate-level time-based power analysis on GB300 (sm_103a).

A thin ctypes binding over ``libpa.so`` (C ABI in ``include/pa.h``). The
functions ``pa_create``, ``pa_load_library``, ``pa_load_netlist``,
``pa_load_events``, ``pa_run``, ``pa_destroy`` and ``pa_last_error`` marshal
arguments only; every step of the computation runs in the library's CUDA
kernels. ``PowerAnalyzer`` wraps them for numpy / torch callers.

There is no CPU fallback: if ``libpa.so`` is missing or cannot be loaded,
importing the binding's entry points raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

PA_OK = 0
PA_ERR_ARG, PA_ERR_ORDER, PA_ERR_UNSORTED, PA_ERR_RANGE = -1, -2, -3, -4
PA_ERR_TOGGLE, PA_ERR_OOM, PA_ERR_CUDA, PA_ERR_INTERNAL = -5, -6, -7, -8
PA_MEM_HOST, PA_MEM_DEVICE = 0, 1
PA_RUN_TIMING, PA_RUN_GLITCH_ALL, PA_RUN_ESW_RISE, PA_RUN_PART_STATS = 1, 2, 4, 8
PA_PART_EVENTS, PA_PART_DENSITY, PA_PART_FIXED = 0, 1, 2
PARTITIONS = {"events": PA_PART_EVENTS, "density": PA_PART_DENSITY, "fixed": PA_PART_FIXED}

ERR_NAMES = {0: "PA_OK", -1: "PA_ERR_ARG", -2: "PA_ERR_ORDER", -3: "PA_ERR_UNSORTED", -4: "PA_ERR_RANGE",
             -5: "PA_ERR_TOGGLE", -6: "PA_ERR_OOM", -7: "PA_ERR_CUDA", -8: "PA_ERR_INTERNAL"}

_vp = ctypes.c_void_p


class PaLibrary(ctypes.Structure):
    _fields_ = [("n_cells", ctypes.c_uint32), ("n_inputs", _vp), ("n_slew", _vp), ("n_load", _vp),
                ("slew_axis", _vp), ("load_axis", _vp), ("lut_off", _vp), ("lut", _vp),
                ("lut_len", ctypes.c_uint64), ("leak_off", _vp), ("leak", _vp), ("leak_len", ctypes.c_uint64)]


class PaNetlist(ctypes.Structure):
    _fields_ = [("n_gates", ctypes.c_uint32), ("cell_id", _vp), ("load_ff", _vp), ("init_in", _vp),
                ("init_out", _vp)]


class PaEvents(ctypes.Structure):
    _fields_ = [("n_pins", ctypes.c_uint64), ("n_events", ctypes.c_uint64), ("pin_off", _vp), ("t_ns", _vp),
                ("slew_ps", _vp), ("value", _vp), ("mem", ctypes.c_int32)]


class PaRunParams(ctypes.Structure):
    _fields_ = [("vdd", ctypes.c_double), ("t_clk_ns", ctypes.c_float), ("n_cycles", ctypes.c_uint32),
                ("t_max_ns", ctypes.c_double), ("tile_events", ctypes.c_uint32),
                ("heavy_events", ctypes.c_uint32), ("flags", ctypes.c_uint32), ("part_mode", ctypes.c_uint32),
                ("n_evt_tgt", ctypes.c_uint32), ("n_thr_floor", ctypes.c_uint32), ("n_cyc_fix", ctypes.c_uint32)]


class PaResult(ctypes.Structure):
    _fields_ = [("p_int_w", ctypes.c_double), ("p_sw_w", ctypes.c_double), ("p_gl_w", ctypes.c_double),
                ("p_leak_w", ctypes.c_double), ("t_max_ns", ctypes.c_double), ("out_mem", ctypes.c_int32),
                ("waveform_w", _vp), ("event_count", _vp), ("glitch_count", _vp), ("state_pre", _vp),
                ("lut_ij", _vp), ("is_glitch", _vp), ("ms_partition", ctypes.c_float),
                ("ms_fused", ctypes.c_float), ("ms_reduce", ctypes.c_float), ("ms_total", ctypes.c_float),
                ("n_tiles", ctypes.c_uint32), ("n_heavy", ctypes.c_uint32), ("kernel_launches", ctypes.c_uint32),
                ("path", ctypes.c_uint32), ("gate_power_w", _vp), ("cell_power_w", _vp),
                ("part_threads", ctypes.c_uint64), ("part_evt_p50", ctypes.c_uint32),
                ("part_evt_p90", ctypes.c_uint32), ("part_evt_p99", ctypes.c_uint32),
                ("part_evt_max", ctypes.c_uint32)]


class PaError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{ERR_NAMES.get(code, code)}: {message}")
        self.code = code


EXPORTS = ("pa_create", "pa_destroy", "pa_load_library", "pa_load_netlist", "pa_load_events", "pa_run",
           "pa_run_noalloc", "pa_run_stream", "pa_build_bands", "pa_default_params", "pa_last_error", "pa_version")
PA_PATH_UNBANDED, PA_PATH_BANDED, PA_PATH_WINDOWS, PA_PATH_WARP = 0, 1, 2, 3
PA_NOALLOC_MAX_CYCLES = 65536
PA_NOALLOC_MAX_GATES = 262144

_lib = None


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libpa.so (raises if it is not built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise ImportError(f"libpa.so is not built ({_build.LIB}); run __graft_entry__.build()")
        L = ctypes.CDLL(_build.LIB)
        L.pa_create.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, _vp]
        L.pa_destroy.argtypes = [_vp]
        L.pa_destroy.restype = None
        L.pa_load_library.argtypes = [_vp, ctypes.POINTER(PaLibrary)]
        L.pa_load_netlist.argtypes = [_vp, ctypes.POINTER(PaNetlist)]
        L.pa_load_events.argtypes = [_vp, ctypes.POINTER(PaEvents)]
        L.pa_run.argtypes = [_vp, ctypes.POINTER(PaRunParams), ctypes.POINTER(PaResult)]
        L.pa_run_noalloc.argtypes = [_vp, ctypes.POINTER(PaRunParams), ctypes.POINTER(PaResult)]
        L.pa_run_stream.argtypes = [_vp, ctypes.POINTER(PaRunParams), ctypes.POINTER(PaEvents), ctypes.c_uint64,
                                    ctypes.POINTER(PaResult)]
        L.pa_build_bands.argtypes = [_vp, ctypes.c_float, ctypes.c_uint32]
        L.pa_default_params.argtypes = [ctypes.POINTER(PaRunParams)]
        L.pa_default_params.restype = None
        L.pa_last_error.argtypes = [_vp]
        L.pa_last_error.restype = ctypes.c_char_p
        L.pa_version.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(ctx, rc):
    if rc != PA_OK:
        msg = load_library().pa_last_error(ctx)
        raise PaError(rc, msg.decode() if msg else "")


# --- same-name wrappers of the C ABI (argument marshalling only) -----------

def pa_create(device: int = 0, stream: int | None = None) -> int:
    ctx = _vp()
    rc = load_library().pa_create(ctypes.byref(ctx), int(device), stream)
    if rc != PA_OK:
        raise PaError(rc, "pa_create failed")
    return ctx.value


def pa_destroy(ctx: int) -> None:
    load_library().pa_destroy(ctx)


def pa_load_library(ctx: int, lib: PaLibrary) -> None:
    _check(ctx, load_library().pa_load_library(ctx, ctypes.byref(lib)))


def pa_load_netlist(ctx: int, nl: PaNetlist) -> None:
    _check(ctx, load_library().pa_load_netlist(ctx, ctypes.byref(nl)))


def pa_load_events(ctx: int, ev: PaEvents) -> None:
    _check(ctx, load_library().pa_load_events(ctx, ctypes.byref(ev)))


def pa_run(ctx: int, params: PaRunParams, result: PaResult) -> None:
    _check(ctx, load_library().pa_run(ctx, ctypes.byref(params), ctypes.byref(result)))


def pa_run_noalloc(ctx: int, params: PaRunParams, result: PaResult) -> None:
    """pa_run without any device allocation (scratch in a fixed 5 MiB device
    array; device output arrays only; limits PA_NOALLOC_MAX_CYCLES and
    PA_NOALLOC_MAX_GATES). For callers that may not allocate at run time."""
    _check(ctx, load_library().pa_run_noalloc(ctx, ctypes.byref(params), ctypes.byref(result)))


def pa_run_stream(ctx: int, params: PaRunParams, events: PaEvents, chunk_events: int, result: PaResult) -> None:
    """pa_run on a trace kept in host memory, streamed through the device in
    chunks of whole gates (copies overlapping the computation)."""
    _check(ctx, load_library().pa_run_stream(ctx, ctypes.byref(params), ctypes.byref(events), int(chunk_events),
                                             ctypes.byref(result)))


def pa_build_bands(ctx: int, t_clk_ns: float, band_cycles: int = 0) -> None:
    _check(ctx, load_library().pa_build_bands(ctx, float(t_clk_ns), int(band_cycles)))


def pa_default_params() -> PaRunParams:
    p = PaRunParams()
    load_library().pa_default_params(ctypes.byref(p))
    return p


def pa_last_error(ctx: int) -> str:
    m = load_library().pa_last_error(ctx)
    return m.decode() if m else ""


def pa_version() -> int:
    return load_library().pa_version()


# --- convenience wrapper -----------------------------------------------------

def _addr(a):
    """Data address of a numpy array or a torch tensor (None passes through)."""
    if a is None:
        return None
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    return a.ctypes.data


def _host(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class PowerAnalyzer:
    """Owns one pa_ctx. Arrays may be numpy (host) or CUDA torch tensors
    (device; events only). Host arrays are copied; nothing is retained."""

    def __init__(self, device: int = 0, stream: int | None = None):
        self.ctx = pa_create(device, stream)
        self.n_cycles = None
        self.n_events = 0
        self.n_gates = 0
        self.n_cells = 0

    def close(self):
        if self.ctx:
            pa_destroy(self.ctx)
            self.ctx = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_library(self, n_inputs, n_slew, n_load, slew_axis, load_axis, lut_off, lut, leak_off, leak):
        keep = [_host(n_inputs, np.uint8), _host(n_slew, np.uint8), _host(n_load, np.uint8),
                _host(slew_axis, np.float32), _host(load_axis, np.float32), _host(lut_off, np.uint32),
                _host(lut, np.float32), _host(leak_off, np.uint32), _host(leak, np.float32)]
        L = PaLibrary(len(keep[0]), *(k.ctypes.data for k in keep[:7]), len(keep[6]),
                      keep[7].ctypes.data, keep[8].ctypes.data, len(keep[8]))
        pa_load_library(self.ctx, L)
        self.n_cells = len(keep[0])

    def load_netlist(self, cell_id, load_ff, init_in, init_out):
        keep = [_host(cell_id, np.uint32), _host(load_ff, np.float32), _host(init_in, np.uint8),
                _host(init_out, np.uint8)]
        pa_load_netlist(self.ctx, PaNetlist(len(keep[0]), *(k.ctypes.data for k in keep)))
        self.n_gates = len(keep[0])

    def load_events(self, pin_off, t_ns, slew_ps, value=None):
        dev = hasattr(t_ns, "is_cuda") and t_ns.is_cuda
        if dev:
            arrs = [pin_off, t_ns, slew_ps, value]
            for a in arrs:
                if a is not None and not a.is_contiguous():
                    raise ValueError("device event arrays must be contiguous")
            n_pins = pin_off.numel() - 1
            n_ev = t_ns.numel()
        else:
            arrs = [_host(pin_off, np.uint64), _host(t_ns, np.float32), _host(slew_ps, np.float32),
                    None if value is None else _host(value, np.uint8)]
            n_pins = len(arrs[0]) - 1
            n_ev = len(arrs[1])
        ev = PaEvents(n_pins, n_ev, _addr(arrs[0]), _addr(arrs[1]), _addr(arrs[2]), _addr(arrs[3]),
                      PA_MEM_DEVICE if dev else PA_MEM_HOST)
        pa_load_events(self.ctx, ev)
        self.n_events = n_ev

    def build_bands(self, t_clk_ns, band_cycles: int = 0):
        """Regroup the loaded events by clock bands for runs at this clock."""
        pa_build_bands(self.ctx, t_clk_ns, band_cycles)

    def load_workload(self, w, with_value: bool = True):
        self.load_library(w.n_inputs, w.n_slew, w.n_load, w.slew_axis, w.load_axis, w.lut_off, w.lut,
                          w.leak_off, w.leak)
        self.load_netlist(w.cell_id, w.load_ff, w.init_in, w.init_out)
        self.load_events(w.pin_off, w.t_ns, w.slew_ps, w.value if with_value else None)

    def run(self, vdd, t_clk_ns, n_cycles, t_max_ns=0.0, tile_events=0, heavy_events=0, timing=False,
            waveform=True, counts=True, debug=False, gate_power=False, cell_power=False, glitch_all=False,
            esw_rise=False, out=None, stream=None, chunk_events=0, partition="events", n_evt_tgt=0,
            n_thr_floor=0, n_cyc_fix=0, part_stats=False):
        """Run the power computation. Returns a dict with ``p_int, p_sw, p_gl,
        p_leak`` (W), ``t_max`` and, as requested, ``waveform`` (f32 W per
        cycle), ``event_count``/``glitch_count`` (u32 per cycle), per-event
        ``state_pre``/``lut_ij``/``is_glitch`` (u8), per-gate ``gate_power``
        (f64 W, [gates, 4]: internal, switching, glitch, leakage), per-cell
        ``cell_power`` (f64 W, [cells, 4]: sums over each cell's gates), and ``ms_*``
        timings. ``glitch_all`` / ``esw_rise`` select the alternative readings
        (PA_RUN_GLITCH_ALL / PA_RUN_ESW_RISE). ``stream = (pin_off, t_ns,
        slew_ps, value)`` (host arrays; value may be None) runs pa_run_stream on
        that trace instead of pa_run on the loaded one, in chunks of about
        ``chunk_events`` events (0 = the library's default).
        ``partition`` = "density" or "fixed" runs the paper's (gate, window)
        thread partition (knobs ``n_evt_tgt``, ``n_thr_floor``, ``n_cyc_fix``;
        0 = the library's defaults); the result then holds ``part_threads`` and,
        with ``part_stats``, ``part_evt`` = (p50, p90, p99, max) events per thread.
        ``out`` may hold preallocated arrays (numpy or CUDA tensors) under the
        same names; CUDA tensors select device output."""
        flags = ((PA_RUN_TIMING if timing else 0) | (PA_RUN_GLITCH_ALL if glitch_all else 0)
                 | (PA_RUN_ESW_RISE if esw_rise else 0) | (PA_RUN_PART_STATS if part_stats else 0))
        p = PaRunParams(float(vdd), float(t_clk_ns), int(n_cycles), float(t_max_ns), int(tile_events),
                        int(heavy_events), flags, PARTITIONS[partition], int(n_evt_tgt), int(n_thr_floor),
                        int(n_cyc_fix))
        r = PaResult()
        res = {}
        out = dict(out or {})
        dev_out = any(hasattr(v, "is_cuda") and v.is_cuda for v in out.values())
        r.out_mem = PA_MEM_DEVICE if dev_out else PA_MEM_HOST

        def arr(name, n, dtype, want):
            if name in out:
                res[name] = out[name]
            elif want and not dev_out:
                res[name] = np.empty(n, dtype)
            else:
                return None
            return _addr(res[name])

        r.waveform_w = arr("waveform", n_cycles, np.float32, waveform)
        r.event_count = arr("event_count", n_cycles, np.uint32, counts)
        r.glitch_count = arr("glitch_count", n_cycles, np.uint32, counts)
        r.state_pre = arr("state_pre", self.n_events, np.uint8, debug)
        r.lut_ij = arr("lut_ij", self.n_events, np.uint8, debug)
        r.is_glitch = arr("is_glitch", self.n_events, np.uint8, debug)
        r.gate_power_w = arr("gate_power", self.n_gates * 4, np.float64, gate_power)
        r.cell_power_w = arr("cell_power", self.n_cells * 4, np.float64, cell_power)
        if stream is None:
            pa_run(self.ctx, p, r)
        else:
            po, tt, ss, vv = stream
            keep = [_host(po, np.uint64), _host(tt, np.float32), _host(ss, np.float32),
                    None if vv is None else _host(vv, np.uint8)]
            ev = PaEvents(len(keep[0]) - 1, len(keep[1]), keep[0].ctypes.data, keep[1].ctypes.data,
                          keep[2].ctypes.data, None if keep[3] is None else keep[3].ctypes.data, PA_MEM_HOST)
            pa_run_stream(self.ctx, p, ev, chunk_events, r)
        for name in ("gate_power", "cell_power"):
            if name in res and not (hasattr(res[name], "is_cuda") and res[name].is_cuda):
                res[name] = np.asarray(res[name]).reshape(-1, 4)
        res.update(p_int=r.p_int_w, p_sw=r.p_sw_w, p_gl=r.p_gl_w, p_leak=r.p_leak_w, t_max=r.t_max_ns,
                   n_tiles=r.n_tiles, n_heavy=r.n_heavy, kernel_launches=r.kernel_launches, path=r.path)
        if r.path == PA_PATH_WINDOWS:
            res["part_threads"] = r.part_threads
            if part_stats:
                res["part_evt"] = (r.part_evt_p50, r.part_evt_p90, r.part_evt_p99, r.part_evt_max)
        if timing:
            res.update(ms_partition=r.ms_partition, ms_fused=r.ms_fused, ms_reduce=r.ms_reduce,
                       ms_total=r.ms_total)
        return res


def build(force: bool = False, verbose: bool = False) -> str:
    return _build.build(force=force, verbose=verbose)
