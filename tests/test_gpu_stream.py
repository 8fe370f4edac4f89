"""pa_run_stream: a trace kept in host memory, streamed through the device in
chunks of whole gates. Parity with the fp64 oracle at the same bar as pa_run
(states are not available on this path), chunk boundaries in the middle of
hot and idle stretches, errors located in the whole trace."""
import numpy as np
import pytest

import oracle
import synth
from tests.test_gpu_gate_power import assert_gate_parity
from tests.test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def glp():
    import gate_level_power_gb300 as glp
    glp.build()
    glp.load_library()
    return glp


def stream_run(glp, w, chunk_events, *, with_value=True, load_trace=False, **kw):
    with glp.PowerAnalyzer(0) as pa:
        pa.load_library(w.n_inputs, w.n_slew, w.n_load, w.slew_axis, w.load_axis, w.lut_off, w.lut, w.leak_off,
                        w.leak)
        pa.load_netlist(w.cell_id, w.load_ff, w.init_in, w.init_out)
        if load_trace:  # a loaded trace is left alone by the streamed run
            pa.load_events(w.pin_off, w.t_ns, w.slew_ps, w.value)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, stream=(w.pin_off, w.t_ns, w.slew_ps,
                                                          w.value if with_value else None),
                   chunk_events=chunk_events, **kw)
        if load_trace:
            r["loaded_run"] = pa.run(w.vdd, w.t_clk_ns, w.n_cycles)
    return r


@pytest.mark.parametrize("cfg,chunk", [(1, 700), (2, 1_000_000), (2, 0), (2, 123_457)])
def test_stream_matches_oracle(glp, cfg, chunk):
    w = synth.generate(cfg)
    r = stream_run(glp, w, chunk)
    o = oracle.run(w, threads=8)
    assert_parity(r, o, debug=False)
    expect = 1 if chunk == 0 else -(-w.n_events // chunk)
    assert r["n_tiles"] >= min(expect, 2)


def test_stream_skewed_hot_gates_larger_than_a_chunk_and_modes(glp):
    # Zipf activity: some gates alone exceed the chunk target (a chunk of one gate)
    w = synth.custom(seed=22, n_gates=20000, n_cells=32, k_mode=1, n_cycles=2000, t_clk_ns=1.0,
                     n_events=3000000, activity=1, zipf_s=1.2, pair_frac=0.1, threads=8)
    assert w.stats["max_gate_events"] > 20000
    r = stream_run(glp, w, 20000, gate_power=True, glitch_all=True, esw_rise=True)
    o = oracle.run(w, threads=8, gate_power=True, glitch_mode=1, esw_mode=1)
    assert_parity(r, o, debug=False)
    assert_gate_parity(r["gate_power"], o["gate_power"])


def test_stream_without_values_and_loaded_trace_untouched(glp):
    w = synth.custom(seed=44, n_gates=60, n_cells=12, k_mode=2, n_slew=5, n_load=4, n_cycles=90, t_clk_ns=1.0,
                     n_events=6000, pair_frac=0.2, quantum_ns=0.125, threads=2)
    r = stream_run(glp, w, 500, with_value=False, load_trace=True)
    o = oracle.run(w, use_value=False)
    assert_parity(r, o, debug=False)
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert r["loaded_run"][key] == pytest.approx(r[key], rel=1e-5)


def test_stream_zero_events(glp):
    w = synth.custom(seed=3, n_gates=500, n_cells=8, n_events=0, n_cycles=20)
    r = stream_run(glp, w, 100)
    o = oracle.run(w)
    assert_parity(r, o, debug=False)


def test_stream_errors_are_located_in_the_whole_trace(glp):
    w = synth.generate(1)
    # an unsorted pair far from the first chunk
    t = w.t_ns.copy()
    pin = int(np.searchsorted(w.pin_off, w.n_events * 3 // 4, side="right") - 1)
    while int(w.pin_off[pin + 1] - w.pin_off[pin]) < 2:
        pin += 1
    e = int(w.pin_off[pin])
    t[e], t[e + 1] = t[e + 1], t[e]
    with glp.PowerAnalyzer(0) as pa:
        pa.load_library(w.n_inputs, w.n_slew, w.n_load, w.slew_axis, w.load_axis, w.lut_off, w.lut, w.leak_off,
                        w.leak)
        pa.load_netlist(w.cell_id, w.load_ff, w.init_in, w.init_out)
        with pytest.raises(glp.PaError) as ei:
            pa.run(w.vdd, w.t_clk_ns, w.n_cycles, stream=(w.pin_off, t, w.slew_ps, w.value), chunk_events=1000)
        assert ei.value.code == glp.PA_ERR_UNSORTED
        assert str(e + 1) in str(ei.value)
        # an event beyond the window
        with pytest.raises(glp.PaError) as ei:
            pa.run(w.vdd, w.t_clk_ns, w.n_cycles // 2, stream=(w.pin_off, w.t_ns, w.slew_ps, w.value),
                   chunk_events=1000)
        assert ei.value.code == glp.PA_ERR_RANGE
        # pin offsets out of order inside a chunk (checked on the device before
        # the chunk is used) and at a chunk boundary (checked on the host)
        po = w.pin_off.copy()
        q = int(np.searchsorted(po, w.n_events // 2))
        while not (po[q - 1] < po[q] < po[q + 1]):
            q += 1
        po[q] = po[q + 1] + 5
        with pytest.raises(glp.PaError) as ei:
            pa.run(w.vdd, w.t_clk_ns, w.n_cycles, stream=(po, w.t_ns, w.slew_ps, w.value), chunk_events=1000)
        assert ei.value.code == glp.PA_ERR_ARG
        po = w.pin_off.copy()
        po[len(po) // 2:] = po[len(po) // 2:] // 3
        po[-1] = w.n_events
        with pytest.raises(glp.PaError) as ei:
            pa.run(w.vdd, w.t_clk_ns, w.n_cycles, stream=(po, w.t_ns, w.slew_ps, w.value), chunk_events=1000)
        assert ei.value.code == glp.PA_ERR_ARG
        # per-event debug arrays are not on this path
        with pytest.raises(glp.PaError) as ei:
            pa.run(w.vdd, w.t_clk_ns, w.n_cycles, debug=True, stream=(w.pin_off, w.t_ns, w.slew_ps, w.value))
        assert ei.value.code == glp.PA_ERR_ARG
        # and the context still runs
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, stream=(w.pin_off, w.t_ns, w.slew_ps, w.value), chunk_events=999)
        o = oracle.run(w)
        assert_parity(r, o, debug=False)


def test_stream_more_than_2_pow_24_events_in_one_cycle(glp):
    # the streamed pass also repeats with integer counts and fp64 bins
    w = synth.custom(seed=31, n_gates=300000, n_cells=8, n_cycles=2, t_clk_ns=1.0, n_events=17_000_000,
                     burst_frac=1.0, burst_width=1, burst_cover=0.5, threads=8)
    r = stream_run(glp, w, 4_000_000)
    o = oracle.run(w, threads=8)
    assert int(o["evcount"].max()) >= 1 << 24
    assert_parity(r, o, debug=False)
