"""GPU parity of the paper's (gate, window) thread partition (pa_run with
part_mode PA_PART_DENSITY / PA_PART_FIXED) against the fp64 oracle.

Bar: the same as every other path (states, LUT intervals, glitch flags and
per-cycle counts bit-exact; totals within 1e-5 relative; waveform bins within
1e-4 of the peak bin; per-gate power within 1e-5 of the gate's total), and the
partition itself -- thread count and the nearest-rank 50th/90th/99th
percentiles and maximum of events per thread -- equal to the partition oracle
(integer results, bit-exact).
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import partition as P
from tests.test_gpu_gate_power import assert_gate_parity
from tests.test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu

MODES = {"density": P.PART_DENSITY, "fixed": P.PART_FIXED}


@pytest.fixture(scope="module")
def glp():
    import gate_level_power_gb300 as glp
    glp.build()
    glp.load_library()
    return glp


def run_part(glp, w, partition, *, n_evt_tgt=0, n_thr_floor=0, n_cyc_fix=0, banded=False, **kw):
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        if banded:  # a built layout does not change what a window run computes
            pa.build_bands(w.t_clk_ns)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, partition=partition, n_evt_tgt=n_evt_tgt,
                   n_thr_floor=n_thr_floor, n_cyc_fix=n_cyc_fix, part_stats=True, **kw)
    assert r["path"] == glp.PA_PATH_WINDOWS
    return r


def assert_partition(r, w, partition, n_evt_tgt=0, n_thr_floor=0, n_cyc_fix=0):
    s = P.stats(w, MODES[partition], n_evt_tgt or 8, n_thr_floor or 1, n_cyc_fix or 1)
    assert r["part_threads"] == s["threads"]
    assert tuple(r["part_evt"]) == (s["p50"], s["p90"], s["p99"], s["max"])


@pytest.mark.parametrize("cfg", [1, 2])
@pytest.mark.parametrize("partition,knobs", [("density", {}), ("density", {"n_evt_tgt": 2, "n_thr_floor": 5}),
                                             ("fixed", {"n_cyc_fix": 8}), ("fixed", {"n_cyc_fix": 1})])
def test_standard_configs(glp, cfg, partition, knobs):
    w = synth.generate(cfg)
    r = run_part(glp, w, partition, debug=True, **knobs)
    o = oracle.run(w, debug=True, threads=8)
    assert_parity(r, o)
    assert_partition(r, w, partition, **knobs)


@pytest.mark.parametrize("seed,quantum,k_mode,t_clk,n_gates,n_events,n_cycles,partition,knobs", [
    (11, 0.0, 1, 1.0, 40, 3000, 50, "density", {}),
    (12, 0.25, 1, 1.0, 40, 3000, 50, "density", {"n_evt_tgt": 3}),     # many cross-pin ties
    (13, 0.125, 2, 0.8, 30, 4000, 40, "fixed", {"n_cyc_fix": 3}),      # all 4-input, non power-of-two clock
    (14, 0.05, 0, 0.8, 200, 6000, 64, "density", {"n_thr_floor": 7}),
    (15, 1.0, 2, 1.0, 20, 2500, 200, "fixed", {"n_cyc_fix": 16}),      # every event on a cycle boundary
    (16, 0.0, 1, 0.3, 300, 20000, 333, "density", {}),
    (17, 0.5, 1, 2.0, 7, 1500, 30, "fixed", {"n_cyc_fix": 1000}),      # one thread per gate
])
def test_tie_heavy_workloads(glp, seed, quantum, k_mode, t_clk, n_gates, n_events, n_cycles, partition, knobs):
    w = synth.custom(seed=seed, n_gates=n_gates, n_cells=12, k_mode=k_mode, n_slew=5, n_load=4,
                     n_cycles=n_cycles, t_clk_ns=t_clk, n_events=n_events, pair_frac=0.2,
                     quantum_ns=quantum, threads=2)
    r = run_part(glp, w, partition, debug=True, **knobs)
    o = oracle.run(w, debug=True)
    assert_parity(r, o)
    assert_partition(r, w, partition, **knobs)


def test_skewed_gates_and_a_built_layout(glp):
    # dense gates (many events of one pin in one cycle) get one-cycle windows
    w = synth.custom(seed=23, n_gates=40, n_cells=8, k_mode=1, n_slew=6, n_load=6, n_cycles=24,
                     t_clk_ns=1.0, n_events=60000, pair_frac=0.1, quantum_ns=0.001, threads=4)
    r = run_part(glp, w, "density", banded=True, debug=True)
    o = oracle.run(w, debug=True, threads=4)
    assert_parity(r, o)
    assert_partition(r, w, "density")
    assert r["part_evt"][3] > 100


@pytest.mark.parametrize("partition", ["density", "fixed"])
def test_gate_and_cell_power(glp, partition):
    w = synth.generate(2)
    r = run_part(glp, w, partition, n_cyc_fix=4, gate_power=True, cell_power=True, debug=False)
    o = oracle.run(w, gate_power=True, threads=8)
    assert_gate_parity(r["gate_power"], o["gate_power"])
    cp = np.zeros((len(w.n_inputs), 4))
    np.add.at(cp, w.cell_id.astype(np.int64), o["gate_power"])
    assert_gate_parity(r["cell_power"], cp)
    assert_parity(r, o, debug=False)


@pytest.mark.parametrize("glitch_all,esw_rise", [(True, False), (False, True), (True, True)])
def test_alternative_readings(glp, glitch_all, esw_rise):
    w = synth.custom(seed=42, n_gates=60, n_cells=12, k_mode=2, n_slew=5, n_load=4, n_cycles=90, t_clk_ns=0.8,
                     n_events=6000, pair_frac=0.2, quantum_ns=0.125, threads=2)
    r = run_part(glp, w, "density", debug=True, glitch_all=glitch_all, esw_rise=esw_rise)
    o = oracle.run(w, debug=True, glitch_mode=int(glitch_all), esw_mode=int(esw_rise))
    assert_parity(r, o)


def test_without_statistics_and_with_timing(glp):
    w = synth.generate(2)
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, partition="density", timing=True)
    o = oracle.run(w, threads=8)
    assert_parity(r, o, debug=False)
    assert "part_evt" not in r
    assert r["part_threads"] == P.stats(w, P.PART_DENSITY)["threads"]
    assert r["ms_fused"] > 0 and r["ms_total"] >= r["ms_fused"]


def test_more_than_2_pow_24_events_in_one_cycle_counts_exactly(glp):
    w = synth.custom(seed=31, n_gates=300000, n_cells=8, n_cycles=2, t_clk_ns=1.0, n_events=17_000_000,
                     burst_frac=1.0, burst_width=1, burst_cover=0.5, threads=8)
    r = run_part(glp, w, "density", debug=False)
    o = oracle.run(w, threads=8)
    assert int(o["evcount"].max()) >= 1 << 24
    assert_parity(r, o, debug=False)


def test_zero_events_and_rejected_modes(glp):
    w = synth.custom(seed=3, n_gates=50, n_cells=4, n_events=0, n_cycles=20, threads=1)
    r = run_part(glp, w, "density", debug=False)
    o = oracle.run(w)
    assert_parity(r, o, debug=False)
    assert r["part_evt"] == (0, 0, 0, 0) and r["part_threads"] == 50
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        p = glp.PaRunParams(float(w.vdd), float(w.t_clk_ns), int(w.n_cycles), 0.0, 0, 0, 0, 3, 0, 0, 0)
        with pytest.raises(glp.PaError) as ei:
            glp.pa_run(pa.ctx, p, glp.PaResult())
        assert ei.value.code == glp.PA_ERR_ARG
        p.part_mode = glp.PA_PART_DENSITY
        with pytest.raises(glp.PaError) as ei:
            glp.pa_run_noalloc(pa.ctx, p, glp.PaResult())
        assert ei.value.code == glp.PA_ERR_ARG
        with pytest.raises(glp.PaError) as ei:
            pa.run(w.vdd, w.t_clk_ns, w.n_cycles, partition="fixed",
                   stream=(w.pin_off, w.t_ns, w.slew_ps, w.value))
        assert ei.value.code == glp.PA_ERR_ARG
