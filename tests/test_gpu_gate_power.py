"""GPU parity of the per-gate power output (pa_result.gate_power_w) against
the fp64 oracle, on the banded and the unbanded kernel.

Bar: every component of every gate (internal, switching, glitch, leakage)
within 1e-5 of that gate's total power; the per-gate sums equal the design
totals within 1e-5; asking for per-gate power leaves the totals, waveform and
counts at their parity bar.
"""
import numpy as np
import pytest

import oracle
import synth
from gate_level_power_gb300 import analysis
from tests.test_gpu_parity import assert_parity, golden

pytestmark = pytest.mark.gpu

TOL_G = 1e-5


@pytest.fixture(scope="module")
def glp():
    import gate_level_power_gb300 as glp
    glp.build()
    glp.load_library()
    return glp


def run_gates(glp, w, banded, *, band_cycles=0, debug=False, out=None):
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        if banded:
            pa.build_bands(w.t_clk_ns, band_cycles)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, debug=debug, gate_power=True, out=out)
    assert r["path"] == (glp.PA_PATH_BANDED if banded else glp.PA_PATH_UNBANDED)
    return r


def assert_gate_parity(g, og):
    g = np.asarray(g, np.float64).reshape(-1, 4)
    assert g.shape == og.shape
    tot = np.abs(og).sum(axis=1, keepdims=True)
    err = np.abs(g - og)
    bad = err > TOL_G * tot + 1e-30
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:5].tolist(), float((err / np.maximum(tot, 1e-300)).max()))


def assert_sums(r):
    g = np.asarray(r["gate_power"], np.float64).reshape(-1, 4)
    for m, key in enumerate(("p_int", "p_sw", "p_gl", "p_leak")):
        assert float(g[:, m].sum()) == pytest.approx(r[key], rel=TOL_G, abs=1e-30), key


@pytest.mark.parametrize("name", ["w1_inverter_glitch.json", "w2_nand2_tie.json"])
@pytest.mark.parametrize("banded", [False, True])
def test_gate_power_golden(glp, name, banded):
    w, d = golden(name)
    r = run_gates(glp, w, banded, band_cycles=1)
    ex = d["expected"]
    for m, key in enumerate(("p_int", "p_sw", "p_gl", "p_leak")):
        assert r["gate_power"][0, m] == pytest.approx(ex[key], rel=TOL_G, abs=1e-30), key


@pytest.mark.parametrize("cfg,banded,bc", [(1, False, 0), (1, True, 8), (2, False, 0), (2, True, 0),
                                           (2, True, 64)])
def test_gate_power_standard_configs(glp, cfg, banded, bc):
    w = synth.generate(cfg)
    r = run_gates(glp, w, banded, band_cycles=bc)
    o = oracle.run(w, gate_power=True, threads=8)
    assert_gate_parity(r["gate_power"], o["gate_power"])
    assert_sums(r)
    assert_parity(r, o, debug=False)
    # the paper's spatial accuracy measures, against the oracle's gate power
    assert analysis.hotspot_overlap(r["gate_power"], o["gate_power"], 0.01) >= 0.99
    assert analysis.rank_correlation(r["gate_power"], o["gate_power"]) >= 0.999


@pytest.mark.parametrize("banded", [False, True])
def test_gate_power_ties_and_pulses_with_debug_arrays(glp, banded):
    # cross-pin ties and glitch pulses; per-event debug arrays asked for as well
    w = synth.custom(seed=42, n_gates=60, n_cells=12, k_mode=2, n_slew=5, n_load=4, n_cycles=90, t_clk_ns=0.8,
                     n_events=6000, pair_frac=0.2, quantum_ns=0.125, threads=2)
    r = run_gates(glp, w, banded, band_cycles=8, debug=True)
    o = oracle.run(w, gate_power=True, debug=True)
    assert_gate_parity(r["gate_power"], o["gate_power"])
    assert_parity(r, o)


def test_gate_power_skewed_with_big_gates(glp):
    # heavy gates: narrow windows in the banded layout, and gates with more
    # than 15 events of a pin in one cycle streamed by the unbanded kernel in
    # the same run
    w = synth.custom(seed=23, n_gates=40, n_cells=8, k_mode=1, n_slew=6, n_load=6, n_cycles=24,
                     t_clk_ns=1.0, n_events=60000, pair_frac=0.1, quantum_ns=0.001, threads=4)
    r = run_gates(glp, w, True)
    assert r["n_heavy"] > 0
    o = oracle.run(w, gate_power=True, threads=4)
    assert_gate_parity(r["gate_power"], o["gate_power"])
    assert_sums(r)


def test_gate_power_device_output_and_zero_event_gates(glp):
    import torch
    w = synth.custom(seed=3, n_gates=500, n_cells=8, n_events=300, n_cycles=20, threads=1)
    gp = torch.full((len(w.cell_id) * 4,), float("nan"), dtype=torch.float64, device="cuda")
    r = run_gates(glp, w, True, out={"gate_power": gp})
    torch.cuda.synchronize()
    got = gp.cpu().numpy().reshape(-1, 4)
    o = oracle.run(w, gate_power=True)
    assert_gate_parity(got, o["gate_power"])
    # gates without events hold their initial state's leakage and nothing else
    assert (o["gate_power"][:, 0] == 0).sum() > 0
    idle = (o["gate_power"][:, :3] == 0).all(axis=1)
    np.testing.assert_allclose(got[idle, 3], o["gate_power"][idle, 3], rtol=1e-6)
    assert (got[idle, :3] == 0).all()


def test_gate_power_through_noalloc_matches_pa_run(glp):
    import torch
    w = synth.generate(1)
    dev = torch.device("cuda", 0)
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        ref = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, gate_power=True)
        for _ in range(2):  # the no-alloc scratch keeps the last call's contents
            gp = torch.full((len(w.cell_id) * 4,), float("nan"), dtype=torch.float64, device=dev)
            p = glp.PaRunParams(float(w.vdd), float(w.t_clk_ns), int(w.n_cycles), 0.0, 0, 0, 0)
            r = glp.PaResult()
            r.out_mem = glp.PA_MEM_DEVICE
            r.gate_power_w = gp.data_ptr()
            torch.cuda.synchronize()
            glp.pa_run_noalloc(pa.ctx, p, r)
            got = gp.cpu().numpy().reshape(-1, 4)
            assert_gate_parity(got, ref["gate_power"])
            assert r.p_int_w == pytest.approx(ref["p_int"], rel=TOL_G)


def oracle_cell_power(w, og):
    cp = np.zeros((len(w.n_inputs), 4))
    np.add.at(cp, w.cell_id.astype(np.int64), og)
    return cp


@pytest.mark.parametrize("banded,with_gates", [(False, True), (True, True), (True, False)])
def test_cell_power_sums_gate_power_by_cell(glp, banded, with_gates):
    w = synth.generate(2)
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        if banded:
            pa.build_bands(w.t_clk_ns)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, gate_power=with_gates, cell_power=True)
    o = oracle.run(w, gate_power=True, threads=8)
    oc = oracle_cell_power(w, o["gate_power"])
    assert_gate_parity(r["cell_power"], oc)
    if with_gates:
        np.testing.assert_allclose(r["cell_power"], oracle_cell_power(w, r["gate_power"]), rtol=1e-9, atol=0)
    for m, key in enumerate(("p_int", "p_sw", "p_gl", "p_leak")):
        assert float(r["cell_power"][:, m].sum()) == pytest.approx(r[key], rel=TOL_G), key


def test_cell_power_streamed_and_device_output(glp):
    import torch
    w = synth.generate(1)
    cp = torch.full((len(w.n_inputs) * 4,), float("nan"), dtype=torch.float64, device="cuda")
    with glp.PowerAnalyzer(0) as pa:
        pa.load_library(w.n_inputs, w.n_slew, w.n_load, w.slew_axis, w.load_axis, w.lut_off, w.lut, w.leak_off,
                        w.leak)
        pa.load_netlist(w.cell_id, w.load_ff, w.init_in, w.init_out)
        pa.run(w.vdd, w.t_clk_ns, w.n_cycles, out={"cell_power": cp}, stream=(w.pin_off, w.t_ns, w.slew_ps, w.value),
               chunk_events=3000)
    torch.cuda.synchronize()
    o = oracle.run(w, gate_power=True)
    assert_gate_parity(cp.cpu().numpy().reshape(-1, 4), oracle_cell_power(w, o["gate_power"]))
