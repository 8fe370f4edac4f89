"""Full-size parity on the large configurations (200M, 1B and 2B events), in
the launch configurations the benchmark times (the unbanded pass, the banded
layout), for the per-event-output variant of the kernels and for the timed
variant the benchmark runs.

The oracle runs over the whole workload with its full per-cycle leakage split
(every gate's intervals over every cycle; about a minute per configuration on
the host's cores) and checks:
  * all four power totals and the per-cycle event and glitch counts (totals
    within 1e-5 relative, counts bit-exact);
  * every waveform bin, within 1e-4 of the peak bin;
  * per-event gate state, LUT interval and glitch flag bit-exact on sampled gate
    blocks, which include the heaviest gates (streamed in windows); the
    oracle's per-event outputs of every event would need the whole trace's
    arrays a second time in host memory.
The oracle's results are kept per configuration, so each runs once per module.
"""
import os

import numpy as np
import pytest

import oracle
import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL_P = 1e-5
TOL_W = 1e-4


@pytest.fixture(scope="module")
def glp():
    import gate_level_power_gb300 as glp
    glp.build()
    return glp


_ORACLE = {}


def oracle_full(cfg, w):
    """The oracle over all of workload ``w`` (config ``cfg``), full waveform;
    computed once per configuration."""
    if cfg not in _ORACLE:
        _ORACLE[cfg] = oracle.run(w, wave="full", threads=os.cpu_count() or 8)
    return _ORACLE[cfg]


def assert_every_bin(res, o, E=None):
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert abs(res[key] - o[key]) <= TOL_P * abs(o[key]), (key, res[key], o[key])
    if E is not None:
        assert int(o["evcount"].sum()) == E
    np.testing.assert_array_equal(res["event_count"].astype(np.uint64), o["evcount"])
    np.testing.assert_array_equal(res["glitch_count"].astype(np.uint64), o["glcount"])
    peak = float(np.abs(o["waveform"]).max())
    err = np.abs(res["waveform"].astype(np.float64) - o["waveform"])
    worst = int(np.argmax(err))
    assert len(err) == len(o["waveform"])
    assert float(err[worst]) <= TOL_W * peak, (worst, float(err[worst]), peak)


def sub_workload(w, pb, g0, g1):
    """Gates [g0, g1) of w as a workload of their own (offsets rebased)."""
    import copy
    p0, p1 = int(pb[g0]), int(pb[g1])
    e0, e1 = int(w.pin_off[p0]), int(w.pin_off[p1])
    s = copy.copy(w)
    s.cell_id, s.load_ff = w.cell_id[g0:g1], w.load_ff[g0:g1]
    s.init_in, s.init_out = w.init_in[g0:g1], w.init_out[g0:g1]
    s.pin_off = w.pin_off[p0:p1 + 1] - w.pin_off[p0]
    s.t_ns, s.slew_ps = w.t_ns[e0:e1], w.slew_ps[e0:e1]
    s.value = w.value[e0:e1]
    return s, e0, e1


@pytest.mark.parametrize("cfg,banded", [(3, False), (3, True), (4, False), (4, True), (5, False), (5, True), (6, False),
                                        (6, True)])
def test_full_size_config(glp, cfg, banded):
    w = synth.generate(cfg)
    E, G, N = w.n_events, w.n_gates, w.n_cycles
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        if banded:
            pa.build_bands(w.t_clk_ns)
        r = pa.run(w.vdd, w.t_clk_ns, N, debug=True, timing=True)
        fast = pa.run(w.vdd, w.t_clk_ns, N, timing=True)  # the timed kernel variant (no per-event outputs)
    assert r["path"] == (glp.PA_PATH_BANDED if banded else glp.PA_PATH_UNBANDED)
    assert fast["path"] == (glp.PA_PATH_BANDED if banded else glp.PA_PATH_WARP)
    assert r["n_heavy"] > 0
    assert r["n_tiles"] > 0 or (cfg == 6 and not banded)  # config 6's gates are all heavy for the unbanded kernel
    # totals, counts and every waveform bin over all gates, for both variants
    o = oracle_full(cfg, w)
    for res in (r, fast):
        assert_every_bin(res, o, E)
    # per-event outputs on sampled gate blocks, heaviest gates included
    rng = np.random.default_rng(cfg)
    pb = w.pin_base().astype(np.int64)
    n_g = np.diff(w.pin_off.astype(np.int64)[pb])
    heavy = np.argsort(n_g)[-12:]
    blocks = [(int(g), int(g) + 1) for g in heavy]
    bs = max(1, min(3000, G // 8, int(2e6 * G / max(1, E))))  # blocks of about 2M events at most
    for b in rng.choice(G - bs, 6, replace=False):
        blocks.append((int(b), int(b) + bs))
    for g0, g1 in blocks:
        s, e0, e1 = sub_workload(w, pb, g0, g1)
        so = oracle.run(s, wave="none", debug=True)
        for key in ("state_pre", "lut_ij", "is_glitch"):
            np.testing.assert_array_equal(r[key][e0:e1], so[key], err_msg=f"{key} gates [{g0}, {g1})")


@pytest.mark.parametrize("partition,knobs", [("density", {}), ("fixed", {"n_cyc_fix": 32})])
def test_full_size_paper_partition(glp, partition, knobs):
    # the paper's (gate, window) thread partition on the large skewed workload
    # (config 3: 26M threads at density, 313M at 32 cycles per thread)
    w = synth.generate(3)
    N = w.n_cycles
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        r = pa.run(w.vdd, w.t_clk_ns, N, partition=partition, **knobs)
    assert r["path"] == glp.PA_PATH_WINDOWS
    assert_every_bin(r, oracle_full(3, w), w.n_events)


def test_full_size_streamed_run(glp):
    # the one-shot path of the benchmark's e2e figure: the 1B-event trace kept
    # in host memory, streamed through the device in chunks
    w = synth.generate(4)
    N = w.n_cycles
    with glp.PowerAnalyzer(0) as pa:
        pa.load_library(w.n_inputs, w.n_slew, w.n_load, w.slew_axis, w.load_axis, w.lut_off, w.lut, w.leak_off,
                        w.leak)
        pa.load_netlist(w.cell_id, w.load_ff, w.init_in, w.init_out)
        r = pa.run(w.vdd, w.t_clk_ns, N, stream=(w.pin_off, w.t_ns, w.slew_ps, w.value))
    assert r["n_tiles"] > 1  # chunks
    assert_every_bin(r, oracle_full(4, w), w.n_events)
