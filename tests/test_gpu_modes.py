"""GPU parity of the alternative readings (run flags PA_RUN_GLITCH_ALL and
PA_RUN_ESW_RISE) against the fp64 oracle in the same modes, on the banded and
the unbanded kernel, with the same bar as the default readings."""
import pytest

import oracle
import synth
from tests.test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu

MODES = [(1, 0), (0, 1), (1, 1)]  # (glitch_mode, esw_mode)


@pytest.fixture(scope="module")
def glp():
    import gate_level_power_gb300 as glp
    glp.build()
    glp.load_library()
    return glp


def run_modes(glp, w, banded, gm, em, with_value=True, band_cycles=0):
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w, with_value=with_value)
        if banded:
            pa.build_bands(w.t_clk_ns, band_cycles)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, debug=True, glitch_all=bool(gm), esw_rise=bool(em))
    assert r["path"] == (glp.PA_PATH_BANDED if banded else glp.PA_PATH_UNBANDED)
    return r


@pytest.mark.parametrize("gm,em", MODES)
@pytest.mark.parametrize("banded", [False, True])
def test_modes_config2(glp, gm, em, banded):
    w = synth.generate(2)
    r = run_modes(glp, w, banded, gm, em)
    o = oracle.run(w, debug=True, threads=8, glitch_mode=gm, esw_mode=em)
    assert_parity(r, o)


@pytest.mark.parametrize("gm,em", MODES)
@pytest.mark.parametrize("banded", [False, True])
def test_modes_ties_pulses_and_values(glp, gm, em, banded):
    w = synth.custom(seed=44, n_gates=60, n_cells=12, k_mode=2, n_slew=5, n_load=4, n_cycles=90, t_clk_ns=1.0,
                     n_events=6000, pair_frac=0.2, quantum_ns=0.125, threads=2)
    for with_value in (True, False):
        r = run_modes(glp, w, banded, gm, em, with_value=with_value, band_cycles=4)
        o = oracle.run(w, debug=True, glitch_mode=gm, esw_mode=em, use_value=with_value)
        assert_parity(r, o)


@pytest.mark.parametrize("m", [2, 8])
def test_modes_stress_waveform_banded(glp, m):
    # every pin toggling m times per cycle: in the glitch-all reading every event is a glitch
    w = synth.generate(6, n_gates=30, n_cycles=120, toggles=m)
    r = run_modes(glp, w, True, 1, 1)
    o = oracle.run(w, debug=True, threads=4, glitch_mode=1, esw_mode=1)
    assert_parity(r, o)
    assert int(r["glitch_count"].sum()) == w.n_events


def test_unknown_flag_is_rejected(glp):
    w = synth.generate(1)
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        p = glp.PaRunParams(float(w.vdd), float(w.t_clk_ns), int(w.n_cycles), 0.0, 0, 0, 16)
        with pytest.raises(glp.PaError) as ei:
            glp.pa_run(pa.ctx, p, glp.PaResult())
        assert ei.value.code == glp.PA_ERR_ARG
