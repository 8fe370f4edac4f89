"""Error paths of the C ABI on a GPU. Every failure here is made on the host
side (bad input arrays, wrong call order, an injected allocation failure);
none faults or hangs the device."""
import os

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def glp():
    import gate_level_power_gb300 as glp
    glp.build()
    return glp


@pytest.fixture()
def w():
    return synth.custom(seed=9, n_gates=30, n_cells=8, n_events=600, n_cycles=20, threads=1)


def loaded(glp, w, upto="netlist"):
    pa = glp.PowerAnalyzer(0)
    pa.load_library(w.n_inputs, w.n_slew, w.n_load, w.slew_axis, w.load_axis, w.lut_off, w.lut, w.leak_off,
                    w.leak)
    if upto in ("netlist", "events"):
        pa.load_netlist(w.cell_id, w.load_ff, w.init_in, w.init_out)
    if upto == "events":
        pa.load_events(w.pin_off, w.t_ns, w.slew_ps, w.value)
    return pa


def expect(glp, code, fn, *a, **k):
    with pytest.raises(glp.PaError) as ei:
        fn(*a, **k)
    assert ei.value.code == code, str(ei.value)
    return str(ei.value)


def test_call_order(glp, w):
    with glp.PowerAnalyzer(0) as pa:
        expect(glp, glp.PA_ERR_ORDER, pa.load_netlist, w.cell_id, w.load_ff, w.init_in, w.init_out)
        expect(glp, glp.PA_ERR_ORDER, pa.load_events, w.pin_off, w.t_ns, w.slew_ps, w.value)
        expect(glp, glp.PA_ERR_ORDER, pa.run, w.vdd, w.t_clk_ns, w.n_cycles)


def _first_multi_event_pin(w):
    d = np.diff(w.pin_off.astype(np.int64))
    p = int(np.nonzero(d >= 2)[0][0])
    return int(w.pin_off[p])


def test_unsorted_events(glp, w):
    t = w.t_ns.copy()
    e = _first_multi_event_pin(w)
    t[e + 1] = t[e]
    with loaded(glp, w) as pa:
        msg = expect(glp, glp.PA_ERR_UNSORTED, pa.load_events, w.pin_off, t, w.slew_ps, w.value)
        assert f"event {e + 1}" in msg
        # the failed load left no events behind
        expect(glp, glp.PA_ERR_ORDER, pa.run, w.vdd, w.t_clk_ns, w.n_cycles)


@pytest.mark.parametrize("bad", [-1.0, float("nan"), float("inf")])
def test_bad_time(glp, w, bad):
    t = w.t_ns.copy()
    t[5] = bad
    with loaded(glp, w) as pa:
        expect(glp, glp.PA_ERR_RANGE, pa.load_events, w.pin_off, t, w.slew_ps, w.value)


@pytest.mark.parametrize("bad", [0.0, -3.0, float("nan")])
def test_bad_slew(glp, w, bad):
    s = w.slew_ps.copy()
    s[7] = bad
    with loaded(glp, w) as pa:
        expect(glp, glp.PA_ERR_RANGE, pa.load_events, w.pin_off, w.t_ns, s, w.value)


def test_non_toggling_value(glp, w):
    v = w.value.copy()
    e = _first_multi_event_pin(w)
    v[e + 1] = v[e]
    with loaded(glp, w) as pa:
        expect(glp, glp.PA_ERR_TOGGLE, pa.load_events, w.pin_off, w.t_ns, w.slew_ps, v)


def test_bad_pin_offsets(glp, w):
    with loaded(glp, w) as pa:
        po = w.pin_off.copy()
        po[3], po[4] = po[4] + 1, po[3]
        expect(glp, glp.PA_ERR_ARG, pa.load_events, po, w.t_ns, w.slew_ps, w.value)
        expect(glp, glp.PA_ERR_ARG, pa.load_events, w.pin_off[:-1], w.t_ns, w.slew_ps, w.value)
        po = w.pin_off.copy()
        po[-1] += 1
        expect(glp, glp.PA_ERR_ARG, pa.load_events, po, w.t_ns, w.slew_ps, w.value)


def test_bad_library_and_netlist(glp, w):
    with glp.PowerAnalyzer(0) as pa:
        sax = w.slew_axis.copy()
        sax[0, 1] = sax[0, 0]
        expect(glp, glp.PA_ERR_ARG, pa.load_library, w.n_inputs, w.n_slew, w.n_load, sax, w.load_axis,
               w.lut_off, w.lut, w.leak_off, w.leak)
        k = w.n_inputs.copy()
        k[0] = 5
        expect(glp, glp.PA_ERR_ARG, pa.load_library, k, w.n_slew, w.n_load, w.slew_axis, w.load_axis,
               w.lut_off, w.lut, w.leak_off, w.leak)
        pa.load_library(w.n_inputs, w.n_slew, w.n_load, w.slew_axis, w.load_axis, w.lut_off, w.lut,
                        w.leak_off, w.leak)
        cid = w.cell_id.copy()
        cid[3] = len(w.n_inputs)
        expect(glp, glp.PA_ERR_RANGE, pa.load_netlist, cid, w.load_ff, w.init_in, w.init_out)
        ld = w.load_ff.copy()
        ld[2] = np.nan
        expect(glp, glp.PA_ERR_RANGE, pa.load_netlist, w.cell_id, ld, w.init_in, w.init_out)


def test_run_parameter_checks(glp, w):
    with loaded(glp, w, "events") as pa:
        expect(glp, glp.PA_ERR_ARG, pa.run, w.vdd, 0.0, w.n_cycles)
        expect(glp, glp.PA_ERR_ARG, pa.run, w.vdd, w.t_clk_ns, 0)
        # fewer cycles than the events span
        expect(glp, glp.PA_ERR_RANGE, pa.run, w.vdd, w.t_clk_ns, w.n_cycles // 2)
        # t_max earlier than the last event
        expect(glp, glp.PA_ERR_RANGE, pa.run, w.vdd, w.t_clk_ns, w.n_cycles, t_max_ns=1.0)
        expect(glp, glp.PA_ERR_ARG, pa.run, w.vdd, w.t_clk_ns, w.n_cycles, tile_events=4000, heavy_events=4000)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles)  # the context is still usable
        assert r["p_leak"] > 0


def test_injected_allocation_failure(glp, w):
    os.environ["PA_TEST_FAIL_ALLOC"] = "2"
    try:
        pa = glp.PowerAnalyzer(0)
    finally:
        del os.environ["PA_TEST_FAIL_ALLOC"]
    with pa:
        expect(glp, glp.PA_ERR_OOM, pa.load_library, w.n_inputs, w.n_slew, w.n_load, w.slew_axis,
               w.load_axis, w.lut_off, w.lut, w.leak_off, w.leak)
        # later allocations succeed again
        pa.load_library(w.n_inputs, w.n_slew, w.n_load, w.slew_axis, w.load_axis, w.lut_off, w.lut,
                        w.leak_off, w.leak)


def test_stage_wait_timeout_is_reported(glp):
    # Test hook PA_TEST_STAGE_TIMEOUT=i: the banded kernel never starts the
    # TMA stage copy of work item i, so the warp's bounded mbarrier wait runs
    # out (after a few ms under the hook). The kernel records a distinct
    # error, stops that warp and returns; nothing faults and nothing spins.
    w = synth.generate(1)
    os.environ["PA_TEST_STAGE_TIMEOUT"] = "3"
    try:
        pa = glp.PowerAnalyzer(0)
    finally:
        del os.environ["PA_TEST_STAGE_TIMEOUT"]
    with pa:
        pa.load_workload(w)
        pa.build_bands(w.t_clk_ns)
        msg = expect(glp, glp.PA_ERR_INTERNAL, pa.run, w.vdd, w.t_clk_ns, w.n_cycles)
        assert "stage wait timed out" in msg and "item 3" in msg, msg
    # the device context is still usable: a context without the hook runs the
    # same layout to the unbanded run's results
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        ref = pa.run(w.vdd, w.t_clk_ns, w.n_cycles)
        pa.build_bands(w.t_clk_ns)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles)
    assert r["path"] == glp.PA_PATH_BANDED
    np.testing.assert_array_equal(r["event_count"], ref["event_count"])
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert abs(r[key] - ref[key]) <= 1e-5 * abs(ref[key]), key
