"""GPU parity of the banded path (pa_build_bands + pa_run at the banding
clock) against the fp64 oracle, with the same bar as the unbanded path:
states, LUT intervals, glitch flags and per-cycle counts bit-exact; totals
within 1e-5; waveform bins within 1e-4 of the peak bin."""
import numpy as np
import pytest

import oracle
import synth
from tests.test_gpu_parity import assert_parity, golden

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def glp():
    import gate_level_power_gb300 as glp
    glp.build()
    glp.load_library()
    return glp


def banded_run(glp, w, band_cycles=0, t_max=0.0, debug=True, with_value=True):
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w, with_value=with_value)
        pa.build_bands(w.t_clk_ns, band_cycles)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, t_max_ns=t_max, debug=debug)
    assert r["path"] == glp.PA_PATH_BANDED
    return r


@pytest.mark.parametrize("name", ["w1_inverter_glitch.json", "w2_nand2_tie.json"])
def test_golden_banded(glp, name):
    w, d = golden(name)
    for bc in (0, 1, 2):
        r = banded_run(glp, w, band_cycles=bc)
        ex = d["expected"]
        for key in ("p_int", "p_sw", "p_gl", "p_leak"):
            assert r[key] == pytest.approx(ex[key], rel=1e-5, abs=1e-30), (bc, key)
        np.testing.assert_array_equal(r["event_count"], ex["evcount"])
        for key in ("state_pre", "lut_ij", "is_glitch"):
            np.testing.assert_array_equal(r[key], ex[key], err_msg=f"{key} bands of {bc}")


@pytest.mark.parametrize("cfg,bc", [(1, 0), (1, 8), (2, 0), (2, 128), (2, 16)])
def test_standard_configs_banded(glp, cfg, bc):
    w = synth.generate(cfg)
    r = banded_run(glp, w, band_cycles=bc)
    o = oracle.run(w, debug=True, threads=8)
    assert_parity(r, o)


@pytest.mark.parametrize("seed,quantum,k_mode,t_clk,bc", [
    (41, 0.25, 1, 1.0, 4), (42, 0.125, 2, 0.8, 8), (43, 0.0, 0, 0.8, 2), (44, 1.0, 2, 1.0, 4),
    (45, 0.05, 1, 0.3, 64),
])
def test_random_tie_heavy_banded(glp, seed, quantum, k_mode, t_clk, bc):
    w = synth.custom(seed=seed, n_gates=60, n_cells=12, k_mode=k_mode, n_slew=5, n_load=4, n_cycles=90,
                     t_clk_ns=t_clk, n_events=6000, pair_frac=0.2, quantum_ns=quantum, threads=2)
    r = banded_run(glp, w, band_cycles=bc)
    o = oracle.run(w, debug=True)
    assert_parity(r, o)


@pytest.mark.parametrize("bc", [0, 32, 8])
def test_heavy_units_and_streaming_banded(glp, bc):
    # few gates with many events: windows narrower than a band
    w = synth.custom(seed=21, n_gates=12, n_cells=8, k_mode=1, n_slew=6, n_load=6, n_cycles=400,
                     t_clk_ns=1.0, n_events=120000, pair_frac=0.1, quantum_ns=0.01, threads=4)
    r = banded_run(glp, w, band_cycles=bc)
    o = oracle.run(w, debug=True, threads=4)
    assert_parity(r, o)
    assert r["n_heavy"] > 0


def test_mixed_light_heavy_skewed_banded(glp):
    w = synth.custom(seed=22, n_gates=20000, n_cells=32, k_mode=1, n_cycles=2000, t_clk_ns=1.0,
                     n_events=3000000, activity=1, zipf_s=1.2, pair_frac=0.1, threads=8)
    r = banded_run(glp, w, band_cycles=256)
    o = oracle.run(w, debug=True, threads=8)
    assert_parity(r, o)
    assert r["n_heavy"] > 0 and r["n_tiles"] > 0


@pytest.mark.parametrize("factor", [2.0, "last"])
def test_t_max_override_banded(glp, factor):
    w = synth.custom(seed=5, n_gates=60, n_cells=8, n_events=2000, n_cycles=30, t_clk_ns=1.0, pair_frac=0.1)
    t_max = float(w.t_ns.max()) if factor == "last" else factor * w.n_cycles * w.t_clk_ns
    r = banded_run(glp, w, band_cycles=4, t_max=t_max)
    o = oracle.run(w, debug=True, t_max=t_max)
    assert_parity(r, o)


def test_zero_events_banded(glp):
    w = synth.custom(seed=3, n_gates=500, n_cells=8, n_events=0, n_cycles=20)
    r = banded_run(glp, w)
    o = oracle.run(w, debug=True)
    assert_parity(r, o)


def test_other_clock_falls_back_to_unbanded(glp):
    w = synth.generate(1)
    o = oracle.run(w, t_clk=0.5, n_cycles=200)
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        pa.build_bands(w.t_clk_ns)
        r = pa.run(w.vdd, 0.5, 200)
        assert r["path"] == glp.PA_PATH_WARP
        for key in ("p_int", "p_sw", "p_gl", "p_leak"):
            assert r[key] == pytest.approx(o[key], rel=1e-5)
        # reloading events drops the bands
        pa.load_events(w.pin_off, w.t_ns, w.slew_ps, w.value)
        assert pa.run(w.vdd, w.t_clk_ns, w.n_cycles)["path"] == glp.PA_PATH_WARP


def test_build_bands_errors(glp):
    w = synth.generate(1)
    with glp.PowerAnalyzer(0) as pa:
        with pytest.raises(glp.PaError) as ei:
            pa.build_bands(1.0)
        assert ei.value.code == glp.PA_ERR_ORDER
        pa.load_workload(w)
        for args in ((0.0, 0), (1.0, 8192), (1.0, 3)):  # t_clk, too wide, not a power of two
            with pytest.raises(glp.PaError) as ei:
                pa.build_bands(*args)
            assert ei.value.code == glp.PA_ERR_ARG


def test_band_count_limit(glp):
    # events up to cycle ~1.1M: one-cycle bands would be more than the layout's
    # 2^20 - 1 (rejected before any allocation); 4096-cycle bands are fine
    w = synth.custom(seed=5, n_gates=5, n_cells=2, n_cycles=(1 << 20) + 50000, n_events=2000, threads=1)
    assert int(np.floor(w.t_ns.astype(np.float32) / np.float32(w.t_clk_ns)).max()) >= (1 << 20)
    o = oracle.run(w, debug=True)
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        with pytest.raises(glp.PaError) as ei:
            pa.build_bands(w.t_clk_ns, 1)
        assert ei.value.code == glp.PA_ERR_ARG
        pa.build_bands(w.t_clk_ns)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, debug=True)
    assert r["path"] == glp.PA_PATH_BANDED
    assert_parity(r, o)


def test_big_gates_banded(glp):
    # more than 15 events of a pin in one cycle: those gates stay out of the
    # banded layout and are streamed by the unbanded kernel in the same run
    w = synth.custom(seed=23, n_gates=40, n_cells=8, k_mode=1, n_slew=6, n_load=6, n_cycles=24,
                     t_clk_ns=1.0, n_events=60000, pair_frac=0.1, quantum_ns=0.001, threads=4)
    r = banded_run(glp, w)
    o = oracle.run(w, debug=True, threads=4)
    assert_parity(r, o)
    assert r["n_heavy"] > 0


def test_more_than_2_pow_24_events_in_one_cycle_banded(glp):
    # the banded pass also repeats with integer counts and fp64 bins
    w = synth.custom(seed=31, n_gates=300000, n_cells=8, n_cycles=2, t_clk_ns=1.0, n_events=17_000_000,
                     burst_frac=1.0, burst_width=1, burst_cover=0.5, threads=8)
    r = banded_run(glp, w, debug=False)
    o = oracle.run(w, threads=8)
    assert int(o["evcount"].max()) >= 1 << 24
    assert_parity(r, o, debug=False)


@pytest.mark.parametrize("m", [1, 2, 4, 8])
def test_stress_waveform_banded(glp, m):
    # every pin toggling m times per cycle: single-cycle windows for m >= 4,
    # and at m = 8 (more than 7 events of a pin in a cycle) single-cycle
    # windows of up to 32 input events
    w = synth.generate(6, n_gates=40, n_cycles=300, toggles=m)
    r = banded_run(glp, w)
    o = oracle.run(w, debug=True, threads=4)
    assert_parity(r, o)
    assert r["n_tiles"] > 0 and r["n_heavy"] > 0
    # the timed kernel: for m >= 2 the items come in runs of one cycle and merge
    # their bin updates per run
    assert_parity(banded_run(glp, w, debug=False), o, debug=False)


@pytest.mark.parametrize("m", [15, 16])
def test_longest_units_banded(glp, m):
    # every pin toggling m times per cycle: at m = 15 the layout's longest
    # units (a 4-input gate's window of one cycle holds 60 input events, so
    # its states carry across rounds of 32 lanes); at m = 16 no gate fits a
    # unit and all are streamed by the unbanded kernel in the same run
    w = synth.generate(6, n_gates=40, n_cycles=60, toggles=m)
    r = banded_run(glp, w)
    o = oracle.run(w, debug=True, threads=4)
    assert_parity(r, o)
    assert r["n_heavy"] > 0
    assert (r["n_tiles"] > 0) == (m == 15)
    assert_parity(banded_run(glp, w, debug=False), o, debug=False)  # the two-rounds-per-lane path


def test_tie_heavy_long_units_banded(glp):
    # 4-input gates with about 9 events per pin per cycle on a 1/16 ns grid:
    # long single-cycle units full of cross-pin ties (the pre-timestamp
    # fix-up), a few pins past 15 events in a cycle (streamed gates)
    w = synth.custom(seed=77, n_gates=30, n_cells=8, k_mode=2, n_slew=5, n_load=4, n_cycles=12, t_clk_ns=1.0,
                     n_events=9000, pair_frac=0.0, quantum_ns=1 / 16, threads=2)
    r = banded_run(glp, w, band_cycles=4)
    o = oracle.run(w, debug=True)
    assert_parity(r, o)
    assert r["n_tiles"] > 0 and r["n_heavy"] > 0
    assert_parity(banded_run(glp, w, band_cycles=4, debug=False), o, debug=False)


def test_large_library_falls_back_to_unbanded(glp):
    # 200 cells: more than the banded kernel stages in shared memory. The
    # layout call succeeds, builds nothing, and the run takes the unbanded
    # path, at the same bar against the oracle.
    w = synth.custom(seed=29, n_gates=3000, n_cells=200, k_mode=1, n_slew=7, n_load=7, n_cycles=120,
                     n_events=60000, pair_frac=0.1, threads=4)
    assert len(w.n_inputs) == 200
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        pa.build_bands(w.t_clk_ns)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, debug=True)
        fast = pa.run(w.vdd, w.t_clk_ns, w.n_cycles)
    assert r["path"] == glp.PA_PATH_UNBANDED  # per-event outputs: the CTA kernel
    assert fast["path"] == glp.PA_PATH_UNBANDED  # more than 64 cells: the CTA kernel
    o = oracle.run(w, debug=True, threads=8)
    assert_parity(r, o)
    assert_parity(fast, o, debug=False)
