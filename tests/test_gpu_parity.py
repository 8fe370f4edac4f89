"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar (fp32 compute): gate states before each event, LUT interval selections,
glitch flags and per-cycle event/glitch counts bit-exact; P_int, P_sw, P_gl,
P_leak within 1e-5 relative; every waveform bin within 1e-4 of the peak bin.
"""
import numpy as np
import pytest

import oracle
import synth
from tests._util import golden

pytestmark = pytest.mark.gpu

TOL_P = 1e-5
TOL_W = 1e-4


@pytest.fixture(scope="module")
def glp():
    import gate_level_power_gb300 as glp
    glp.build()
    glp.load_library()
    return glp


def gpu_run(glp, w, *, with_value=True, t_max=0.0, debug=True, **kw):
    """One run; with debug, the per-event-output run (CTA kernel), with the
    same run without per-event outputs (the warp kernel, where it applies)
    under ``"fast"``, which assert_parity checks too."""
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w, with_value=with_value)
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, t_max_ns=t_max, debug=debug, **kw)
        if debug:
            r["fast"] = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, t_max_ns=t_max, **kw)
    return r


def assert_parity(r, o, debug=True):
    if "fast" in r:
        assert_parity(r["fast"], o, debug=False)
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert abs(r[key] - o[key]) <= TOL_P * abs(o[key]) + 1e-30, (key, r[key], o[key])
    peak = float(np.abs(o["waveform"]).max())
    err = float(np.abs(r["waveform"].astype(np.float64) - o["waveform"]).max())
    assert err <= TOL_W * peak, (err, peak)
    np.testing.assert_array_equal(r["event_count"].astype(np.uint64), o["evcount"])
    np.testing.assert_array_equal(r["glitch_count"].astype(np.uint64), o["glcount"])
    if debug:
        for key in ("state_pre", "lut_ij", "is_glitch"):
            np.testing.assert_array_equal(r[key], o[key], err_msg=key)


@pytest.mark.parametrize("name", ["w1_inverter_glitch.json", "w2_nand2_tie.json"])
def test_golden_examples_on_gpu(glp, name):
    w, d = golden(name)
    r = gpu_run(glp, w)
    ex = d["expected"]
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert r[key] == pytest.approx(ex[key], rel=TOL_P, abs=1e-30), key
    np.testing.assert_allclose(r["waveform"], ex["waveform"], rtol=0, atol=TOL_W * max(ex["waveform"]))
    np.testing.assert_array_equal(r["event_count"], ex["evcount"])
    np.testing.assert_array_equal(r["glitch_count"], ex["glcount"])
    for key in ("state_pre", "lut_ij", "is_glitch"):
        np.testing.assert_array_equal(r[key], ex[key], err_msg=key)


@pytest.mark.parametrize("cfg", [1, 2])
def test_standard_configs_elementwise(glp, cfg):
    w = synth.generate(cfg)
    r = gpu_run(glp, w)
    o = oracle.run(w, debug=True, threads=8)
    assert_parity(r, o)


@pytest.mark.parametrize("seed,quantum,k_mode,t_clk,n_gates,n_events,n_cycles", [
    (11, 0.0, 1, 1.0, 40, 3000, 50),
    (12, 0.25, 1, 1.0, 40, 3000, 50),      # many cross-pin ties
    (13, 0.125, 2, 0.8, 30, 4000, 40),     # all 4-input, non power-of-two clock
    (14, 0.05, 0, 0.8, 200, 6000, 64),
    (15, 1.0, 2, 1.0, 20, 2500, 200),      # every event on a cycle boundary
    (16, 0.0, 1, 0.3, 300, 20000, 333),
    (17, 0.5, 1, 2.0, 7, 1500, 30),
])
def test_random_tie_heavy_workloads(glp, seed, quantum, k_mode, t_clk, n_gates, n_events, n_cycles):
    w = synth.custom(seed=seed, n_gates=n_gates, n_cells=12, k_mode=k_mode, n_slew=5, n_load=4,
                     n_cycles=n_cycles, t_clk_ns=t_clk, n_events=n_events, pair_frac=0.2,
                     quantum_ns=quantum, threads=2)
    r = gpu_run(glp, w)
    o = oracle.run(w, debug=True)
    assert_parity(r, o)


@pytest.mark.parametrize("tile,heavy", [(0, 0), (64, 64), (2048, 32), (1, 1), (4000, 96)])
def test_heavy_streaming_and_partition_invariance(glp, tile, heavy):
    # few gates, many events: every gate is streamed in windows; ties and glitch pulses
    w = synth.custom(seed=21, n_gates=12, n_cells=8, k_mode=1, n_slew=6, n_load=6, n_cycles=400,
                     t_clk_ns=1.0, n_events=120000, pair_frac=0.1, quantum_ns=0.01, threads=4)
    r = gpu_run(glp, w, tile_events=tile, heavy_events=heavy)
    o = oracle.run(w, debug=True, threads=4)
    assert_parity(r, o)
    if heavy in (1, 32, 64, 96):
        assert r["n_heavy"] > 0


@pytest.mark.parametrize("tile,heavy", [(0, 0), (64, 64), (3000, 1000), (1, 4095)])
def test_partition_invariance_mid(glp, tile, heavy):
    w = synth.generate(2)
    r = gpu_run(glp, w, tile_events=tile, heavy_events=heavy)
    o = oracle.run(w, debug=True, threads=8)
    assert_parity(r, o)


def test_zero_events_gives_constant_leakage(glp):
    w = synth.custom(seed=3, n_gates=500, n_cells=8, n_events=0, n_cycles=20)
    r = gpu_run(glp, w)
    o = oracle.run(w, debug=True)
    assert_parity(r, o)
    assert r["p_int"] == r["p_sw"] == r["p_gl"] == 0.0
    np.testing.assert_allclose(r["waveform"], o["p_leak"], rtol=1e-6)


def test_sparse_gates_with_empty_pins(glp):
    # far more pins than events: most gates and pins have no events
    w = synth.custom(seed=4, n_gates=5000, n_cells=16, n_events=700, n_cycles=77, t_clk_ns=0.8)
    r = gpu_run(glp, w)
    o = oracle.run(w, debug=True)
    assert_parity(r, o)


@pytest.mark.parametrize("factor", [2.0, 1.0, "last"])
def test_t_max_override(glp, factor):
    w = synth.custom(seed=5, n_gates=60, n_cells=8, n_events=2000, n_cycles=30, t_clk_ns=1.0, pair_frac=0.1)
    t_max = float(w.t_ns.max()) if factor == "last" else factor * w.n_cycles * w.t_clk_ns
    r = gpu_run(glp, w, t_max=t_max)
    o = oracle.run(w, debug=True, t_max=t_max)
    assert_parity(r, o)


def test_value_array_optional(glp):
    w = synth.generate(1)
    a = gpu_run(glp, w, with_value=True)
    b = gpu_run(glp, w, with_value=False)
    for key in ("state_pre", "lut_ij", "is_glitch", "event_count", "glitch_count"):
        np.testing.assert_array_equal(a[key], b[key])


def test_repeated_runs_integer_outputs_identical(glp):
    w = synth.generate(2)
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        runs = [pa.run(w.vdd, w.t_clk_ns, w.n_cycles, debug=True) for _ in range(3)]
    for r in runs[1:]:
        for key in ("event_count", "glitch_count", "state_pre", "lut_ij", "is_glitch"):
            np.testing.assert_array_equal(r[key], runs[0][key])
        for key in ("p_int", "p_sw", "p_gl", "p_leak"):
            assert r[key] == pytest.approx(runs[0][key], rel=1e-6)


def test_device_inputs_and_outputs(glp):
    import torch
    w = synth.generate(2)
    o = oracle.run(w, debug=False, threads=8)
    dev = torch.device("cuda", 0)
    po = torch.from_numpy(w.pin_off.view(np.int64)).to(dev)
    t = torch.from_numpy(w.t_ns).to(dev)
    s = torch.from_numpy(w.slew_ps).to(dev)
    v = torch.from_numpy(w.value).to(dev)
    out = dict(waveform=torch.empty(w.n_cycles, dtype=torch.float32, device=dev),
               event_count=torch.empty(w.n_cycles, dtype=torch.int32, device=dev),
               glitch_count=torch.empty(w.n_cycles, dtype=torch.int32, device=dev))
    with glp.PowerAnalyzer(0) as pa:
        pa.load_library(w.n_inputs, w.n_slew, w.n_load, w.slew_axis, w.load_axis, w.lut_off, w.lut,
                        w.leak_off, w.leak)
        pa.load_netlist(w.cell_id, w.load_ff, w.init_in, w.init_out)
        torch.cuda.synchronize()  # the library's stream does not wait on torch's
        pa.load_events(po, t, s, v)
        del po, t, s, v  # the library keeps its own copies
        r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, out=out)
    r["waveform"] = out["waveform"].cpu().numpy()
    r["event_count"] = out["event_count"].cpu().numpy().view(np.uint32)
    r["glitch_count"] = out["glitch_count"].cpu().numpy().view(np.uint32)
    assert_parity(r, o, debug=False)


def test_timing_and_work_counts_reported(glp):
    w = synth.generate(2)
    r = gpu_run(glp, w, debug=False, timing=True)
    assert r["ms_fused"] > 0 and r["ms_total"] >= r["ms_fused"]
    assert r["path"] == glp.PA_PATH_WARP
    # partition (count, scan, emit, piece cut points), fused kernel, final reduction (2)
    assert r["n_tiles"] > 0 and r["kernel_launches"] == 7


def test_more_than_2_pow_24_events_in_one_cycle_counts_exactly(glp):
    # per-cycle counts travel as f32 in the one-per-event vector reduction; a
    # cycle with 2^24 or more events makes the pass repeat with integer counts
    w = synth.custom(seed=31, n_gates=300000, n_cells=8, n_cycles=2, t_clk_ns=1.0, n_events=17_000_000,
                     burst_frac=1.0, burst_width=1, burst_cover=0.5, threads=8)
    r = gpu_run(glp, w, debug=False)
    o = oracle.run(w, threads=8)
    assert int(o["evcount"].max()) >= 1 << 24
    assert_parity(r, o, debug=False)
