"""Pins for the fp64 oracle, against things other than itself: hand-derived
worked examples, closed forms, invariants and an independent brute-force
formulation. CPU only.

Paper: "GPU-Accelerated Gate-Level Time-Based Power Analysis via Event-Density-
Aware Partitioning and Kernel Fusion", Sections 2.4.1-2.4.2, Eqs. 1-4, Figs. 2,
3 and 7.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from tests._util import brute_force, golden, pin_base, workload


def _run(w, **kw):
    kw.setdefault("t_max", getattr(w, "t_max_ns", 0.0))
    return oracle.run(w, debug=True, **kw)


@pytest.mark.parametrize("name", ["w1_inverter_glitch.json", "w2_nand2_tie.json"])
def test_golden_worked_examples(name):
    w, d = golden(name)
    r = _run(w)
    ex = d["expected"]
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert r[key] == pytest.approx(ex[key], rel=1e-12, abs=1e-18), key
    np.testing.assert_allclose(r["waveform"], ex["waveform"], rtol=1e-12, atol=1e-18)
    np.testing.assert_array_equal(r["evcount"], ex["evcount"])
    np.testing.assert_array_equal(r["glcount"], ex["glcount"])
    for key in ("state_pre", "lut_ij", "is_glitch"):
        np.testing.assert_array_equal(r[key], ex[key], err_msg=key)


def _one_gate(k, leak, lut_const=None, lut=None, C=5.0, init_in=0, init_out=0, events=(), n_cycles=10,
              t_clk=1.0, vdd=1.0, slew_axis=(10, 100), load_axis=(1, 100), value=True):
    """events: list per pin of [(t, slew), ...]"""
    ns, nl = len(slew_axis), len(load_axis)
    if lut is None:
        lut = [lut_const[S] for S in range(1 << k) for _ in range(ns * nl)]
    pin_off = [0]
    t, s, v = [], [], []
    for q, evs in enumerate(events):
        init = (init_in >> q) & 1 if q < k else init_out
        for i, (tt, ss) in enumerate(evs):
            t.append(tt); s.append(ss); v.append(init ^ ((i + 1) & 1))
        pin_off.append(len(t))
    pad = lambda a: list(a) + [0] * (8 - len(a))
    return workload(
        dict(n_inputs=[k], n_slew=[ns], n_load=[nl], slew_axis=[pad(slew_axis)], load_axis=[pad(load_axis)],
             lut_off=[0], lut=lut, leak_off=[0], leak=leak),
        dict(cell_id=[0], load_ff=[C], init_in=[init_in], init_out=[init_out]),
        dict(pin_off=pin_off, t_ns=t, slew_ps=s, value=v if value else None),
        dict(vdd=vdd, t_clk_ns=t_clk, n_cycles=n_cycles))


def test_no_events_constant_leakage():
    # Eq. 4 with one interval [0, t_max): P_leak = p_leak(S0), every bin = p_leak(S0).
    w = _one_gate(2, leak=[3.0, 5.0, 7.0, 11.0], lut_const=[1, 1, 1, 1], init_in=2, events=([], [], []))
    r = _run(w)
    assert r["p_leak"] == pytest.approx(7.0e-9, rel=1e-14)
    np.testing.assert_allclose(r["waveform"], 7.0e-9, rtol=1e-14)
    assert r["p_int"] == r["p_sw"] == r["p_gl"] == 0.0


def test_single_toggle_closed_form():
    # one input toggle at t: P_leak = (p0 t + p1 (t_max - t)) / t_max
    t = 3.375
    w = _one_gate(1, leak=[4.0, 9.0], lut_const=[2, 6], events=([(t, 30.0)], []), n_cycles=10)
    r = _run(w)
    assert r["p_leak"] == pytest.approx((4.0 * t + 9.0 * (10 - t)) / 10 * 1e-9, rel=1e-14)
    # the split bin: the event's 2 fJ, plus 0.375 ns at p0 and 0.625 ns at p1
    assert r["waveform"][3] == pytest.approx(2e-6 + (4.0 * 0.375 + 9.0 * 0.625) * 1e-9, rel=1e-13)
    assert r["waveform"][2] == pytest.approx(4.0e-9) and r["waveform"][4] == pytest.approx(9.0e-9)
    # internal energy from the pre-event state's table (state 0 -> 2 fJ)
    assert r["p_int"] == pytest.approx(2.0 / 10 * 1e-6, rel=1e-14)


@pytest.mark.parametrize("n", [1, 2, 5])
def test_lone_output_toggles_closed_form(n):
    # n toggles of a lone output in distinct cycles: P_sw = n * C V^2 / 2 / t_max, no glitches
    C, V = 7.0, 0.8
    evs = [(c + 0.25, 20.0) for c in range(n)]
    w = _one_gate(1, leak=[0.0, 0.0], lut_const=[0, 0], C=C, vdd=V, events=([], evs), n_cycles=8)
    r = _run(w)
    assert r["p_sw"] == pytest.approx(n * 0.5 * C * V * V / 8 * 1e-6, rel=1e-14)
    assert r["p_gl"] == 0 and r["glcount"].sum() == 0 and r["evcount"].sum() == n


@pytest.mark.parametrize("n", [2, 3, 6])
def test_n_events_one_pin_one_cycle_gives_n_minus_1_glitches(n):
    evs = [(2.0 + 0.1 * i, 50.0) for i in range(n)]
    w = _one_gate(1, leak=[0.0, 0.0], lut_const=[0, 0], C=4.0, events=([], evs), n_cycles=4)
    r = _run(w)
    assert r["glcount"][2] == n - 1 and r["evcount"][2] == n
    np.testing.assert_array_equal(r["is_glitch"], [0] + [1] * (n - 1))


def test_glitch_ratio_exact_and_saturation():
    # Eq. 2 reading: r = min(1, pw / mean slew). pw = 31.25 ps, slews 40 / 85 -> r = 0.5
    C, V = 4.0, 1.0
    esw = 0.5 * C * V * V
    w = _one_gate(1, leak=[0.0, 0.0], lut_const=[0, 0], C=C, vdd=V,
                  events=([], [(1.5, 40.0), (1.53125, 85.0)]), n_cycles=4)
    r = _run(w)
    assert r["e_gl"] == pytest.approx(0.5 * esw, rel=1e-14)
    assert r["e_sw"] == pytest.approx(esw, rel=1e-14)
    # wide pulse (500 ps vs 50 ps mean slew) saturates at 1
    w = _one_gate(1, leak=[0.0, 0.0], lut_const=[0, 0], C=C, vdd=V,
                  events=([], [(1.25, 50.0), (1.75, 50.0)]), n_cycles=4)
    r = _run(w)
    assert r["e_gl"] == pytest.approx(esw, rel=1e-14)
    # same pulse straddling a cycle boundary is not a glitch
    w = _one_gate(1, leak=[0.0, 0.0], lut_const=[0, 0], C=C, vdd=V,
                  events=([], [(1.96875, 50.0), (2.03125, 50.0)]), n_cycles=4)
    r = _run(w)
    assert r["e_gl"] == 0.0 and r["e_sw"] == pytest.approx(2 * esw)


@pytest.mark.parametrize("n,init_out", [(1, 0), (2, 0), (5, 0), (5, 1), (4, 1)])
def test_rise_only_switching_closed_form(n, init_out):
    # Eq. 1 alternative: C V^2 per rising output transition, none per falling;
    # n toggles from init_out rise ceil(n/2) (from 0) or floor(n/2) (from 1) times
    C, V = 7.0, 0.8
    evs = [(c + 0.25, 20.0) for c in range(n)]
    w = _one_gate(1, leak=[0.0, 0.0], lut_const=[0, 0], C=C, vdd=V, init_out=init_out, events=([], evs),
                  n_cycles=8)
    rises = (n + 1) // 2 if init_out == 0 else n // 2
    for use_value in (True, False):
        r = oracle.run(w, esw_mode=1, use_value=use_value)
        assert r["p_sw"] == pytest.approx(rises * C * V * V / 8 * 1e-6, rel=1e-14, abs=1e-30)
    # and the totals over a rise/fall pair equal the default reading's
    w2 = _one_gate(1, leak=[0.0, 0.0], lut_const=[0, 0], C=C, vdd=V, events=([], [(0.25, 20.0), (1.25, 20.0)]),
                   n_cycles=8)
    assert oracle.run(w2, esw_mode=1)["p_sw"] == pytest.approx(oracle.run(w2)["p_sw"], rel=1e-14)


@pytest.mark.parametrize("n", [2, 3, 6])
def test_glitch_all_mode_marks_every_event_of_a_multi_event_cycle(n):
    evs = [(2.0 + 0.1 * i, 50.0) for i in range(n)] + [(3.5, 50.0)]
    w = _one_gate(1, leak=[0.0, 0.0], lut_const=[0, 0], C=4.0, events=([], evs), n_cycles=5)
    r = oracle.run(w, debug=True, glitch_mode=1)
    assert r["glcount"][2] == n and r["glcount"][3] == 0 and r["evcount"].sum() == n + 1
    np.testing.assert_array_equal(r["is_glitch"], [1] * n + [0])


def test_glitch_all_mode_ratio_of_the_first_edge():
    # the first event of the cycle takes the pulse it opens: width to the next
    # event, slews of both; pw = 31.25 ps, slews 40 / 85 -> r = 0.5 for both edges
    C, V = 4.0, 1.0
    esw = 0.5 * C * V * V
    w = _one_gate(1, leak=[0.0, 0.0], lut_const=[0, 0], C=C, vdd=V,
                  events=([], [(1.5, 40.0), (1.53125, 85.0)]), n_cycles=4)
    r = oracle.run(w, glitch_mode=1)
    assert r["e_gl"] == pytest.approx(2 * 0.5 * esw, rel=1e-14) and r["e_sw"] == 0.0


def test_bilinear_reproduces_plane_inside_and_outside_axes():
    # a bilinear surface a + b s + c l + d s l is reproduced exactly by bilinear
    # interpolation on any grid, also when extrapolating (slew/load transposed fails)
    # dyadic axes and coefficients: every table value is exact in f32
    sax = [4.0, 12.0, 40.0, 88.0, 296.0]
    lax = [1.0, 3.0, 9.0, 49.0]
    a, b, c, d = 0.5, 1.0 / 64, 0.25, 1.0 / 1024
    lut = [a + b * s + c * l + d * s * l for S in range(2) for s in sax for l in lax]
    for slew, C in [(7.0, 2.0), (41.0, 48.5), (2.0, 0.5), (400.0, 80.0), (4.0, 1.0), (296.0, 49.0)]:
        w = _one_gate(1, leak=[0.0, 0.0], lut=lut, C=C, events=([(0.5, slew)], []), n_cycles=2,
                      slew_axis=sax, load_axis=lax)
        r = _run(w)
        expect = a + b * slew + c * C + d * slew * C
        assert r["e_int"] == pytest.approx(expect, rel=1e-12), (slew, C)
        i = max([m for m in range(len(sax) - 1) if sax[m] <= slew] + [0])
        j = max([m for m in range(len(lax) - 1) if lax[m] <= C] + [0])
        assert r["lut_ij"][0] == (i << 4) | j


def test_grid_point_returns_table_value():
    sax, lax = [10.0, 20.0, 40.0], [1.0, 2.0, 4.0]
    rng = np.random.default_rng(1)
    lut = list(rng.uniform(1, 9, size=2 * 9))
    for i, s in enumerate(sax):
        for j, C in enumerate(lax):
            w = _one_gate(1, leak=[0.0, 0.0], lut=lut, C=C, events=([(0.5, s)], []), n_cycles=1,
                          slew_axis=sax, load_axis=lax)
            assert _run(w)["e_int"] == pytest.approx(np.float32(lut[i * 3 + j]), rel=1e-15)


def test_t_max_override_extends_leakage_and_rescales():
    w = _one_gate(1, leak=[4.0, 9.0], lut_const=[2, 6], events=([(3.0, 30.0)], []), n_cycles=5)
    r = _run(w, t_max=20.0)
    assert r["p_leak"] == pytest.approx((4.0 * 3 + 9.0 * 17) / 20 * 1e-9, rel=1e-14)
    assert r["p_int"] == pytest.approx(2.0 / 20 * 1e-6, rel=1e-14)
    # bins still cover only [0, 5 ns): the event's 2 fJ plus leakage over 5 ns
    assert r["waveform"].sum() * 1.0 == pytest.approx(2e-6 + (4.0 * 3 + 9.0 * 2) * 1e-9, rel=1e-13)


def _invariants(w, r, t_max):
    E = len(w.t_ns)
    assert int(r["evcount"].sum()) == E
    # glitches: per (pin, cycle) run of n events gives n - 1, counted independently here
    cyc = np.floor(w.t_ns.astype(np.float32) / np.float32(w.t_clk_ns)).astype(np.int64)
    pin = np.repeat(np.arange(len(w.pin_off) - 1), np.diff(w.pin_off.astype(np.int64)))
    key = pin * (w.n_cycles + 1) + cyc
    _, counts = np.unique(key, return_counts=True)
    assert int(r["glcount"].sum()) == int((counts - 1).sum())
    tot = r["p_int"] + r["p_sw"] + r["p_gl"] + r["p_leak"]
    assert r["waveform"].sum() * w.t_clk_ns == pytest.approx(tot * t_max, rel=1e-12)


@pytest.mark.parametrize("cfg", [1, 2])
def test_invariants_standard_configs(cfg):
    w = synth.generate(cfg)
    r = oracle.run(w, threads=4)
    _invariants(w, r, w.n_cycles * w.t_clk_ns)


def test_thread_count_and_value_array_do_not_change_results():
    w = synth.generate(1)
    a = oracle.run(w, threads=1, debug=True)
    b = oracle.run(w, threads=7, debug=True, use_value=False)
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert a[key] == pytest.approx(b[key], rel=1e-13)
    np.testing.assert_allclose(a["waveform"], b["waveform"], rtol=1e-12, atol=1e-20)
    for key in ("evcount", "glcount", "state_pre", "lut_ij", "is_glitch"):
        np.testing.assert_array_equal(a[key], b[key])


def _tiny_random(seed, quantum, k_mode=1, pair_frac=0.2, n_gates=6, n_events=120, n_cycles=12, t_clk=1.0):
    return synth.custom(seed=seed, n_gates=n_gates, n_cells=8, k_mode=k_mode, n_slew=4, n_load=3,
                        n_cycles=n_cycles, t_clk_ns=t_clk, n_events=n_events, pair_frac=pair_frac,
                        quantum_ns=quantum, threads=1)


@pytest.mark.parametrize("seed,quantum,k_mode,t_clk", [
    (1, 0.0, 1, 1.0), (2, 0.25, 1, 1.0), (3, 0.125, 2, 1.0), (4, 0.1, 1, 0.8), (5, 0.5, 2, 0.8),
    (6, 0.0, 0, 0.8), (7, 0.05, 1, 1.0),
])
def test_oracle_matches_brute_force(seed, quantum, k_mode, t_clk):
    w = _tiny_random(seed, quantum, k_mode=k_mode, t_clk=t_clk)
    r = oracle.run(w, debug=True)
    b = brute_force(w)
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert r[key] == pytest.approx(b[key], rel=1e-11, abs=1e-22), key
    np.testing.assert_allclose(r["wave_energy"], b["wave_energy"], rtol=1e-10, atol=1e-14)
    np.testing.assert_array_equal(r["evcount"], b["evcount"])
    np.testing.assert_array_equal(r["glcount"], b["glcount"])
    for key in ("state_pre", "lut_ij", "is_glitch"):
        np.testing.assert_array_equal(r[key].astype(np.int64), b[key], err_msg=key)


@pytest.mark.parametrize("seed,quantum,k_mode", [(1, 0.0, 1), (3, 0.125, 2), (6, 0.0, 0)])
def test_per_gate_power_matches_brute_force(seed, quantum, k_mode):
    # per-gate power: each gate's own energies over t_max, against the brute
    # force's per-gate tally (a different formulation of the same quantities)
    w = _tiny_random(seed, quantum, k_mode=k_mode)
    r = oracle.run(w, gate_power=True)
    b = brute_force(w)
    scale = float(np.abs(b["gate_power"]).max())
    np.testing.assert_allclose(r["gate_power"], b["gate_power"], rtol=1e-10, atol=1e-12 * scale)
    assert (b["gate_power"][:, 0] > 0).sum() > 1 and (b["gate_power"][:, 2] > 0).any()


@pytest.mark.parametrize("cfg", [1, 2])
def test_per_gate_power_sums_to_totals(cfg):
    w = synth.generate(cfg)
    r = oracle.run(w, gate_power=True, threads=4)
    for m, key in enumerate(("p_int", "p_sw", "p_gl", "p_leak")):
        assert float(r["gate_power"][:, m].sum()) == pytest.approx(r[key], rel=1e-12), key
    # a gate range walks only its gates, with the same per-gate values
    G = len(w.cell_id)
    part = oracle.run(w, gate_power=True, gate_range=(G // 3, G // 2))
    np.testing.assert_array_equal(part["gate_power"], r["gate_power"][G // 3:G // 2])


def test_per_gate_power_lone_gate_is_the_totals():
    w, d = golden("w1_inverter_glitch.json")
    r = oracle.run(w, gate_power=True)
    assert r["gate_power"].shape == (1, 4)
    for m, key in enumerate(("p_int", "p_sw", "p_gl", "p_leak")):
        assert r["gate_power"][0, m] == pytest.approx(d["expected"][key], rel=1e-12), key


@pytest.mark.parametrize("m", [1, 2, 4, 8])
def test_stress_waveform_counts_closed_form(m):
    # the waveform-bin stress workload: every pin toggles m times in every
    # cycle, so each cycle holds m events per pin and, by the counter reading,
    # m - 1 glitches per pin; bins still sum to the totals
    w = synth.generate(6, n_gates=30, n_cycles=40, toggles=m)
    P = w.n_pins
    assert w.n_events == m * P * w.n_cycles
    r = oracle.run(w)
    assert (r["evcount"] == m * P).all()
    assert (r["glcount"] == (m - 1) * P).all()
    assert (r["p_gl"] > 0) == (m > 1)
    e_tot = r["e_int"] + r["e_sw"] + r["e_gl"] + r["e_leak"]
    assert float(r["wave_energy"].sum()) == pytest.approx(e_tot, rel=1e-12)


@pytest.mark.parametrize("seed,quantum,k_mode,glitch_mode,esw_mode", [
    (2, 0.25, 1, 1, 0), (3, 0.125, 2, 0, 1), (7, 0.05, 1, 1, 1),
])
def test_oracle_modes_match_brute_force(seed, quantum, k_mode, glitch_mode, esw_mode):
    w = _tiny_random(seed, quantum, k_mode=k_mode)
    r = oracle.run(w, debug=True, glitch_mode=glitch_mode, esw_mode=esw_mode)
    b = brute_force(w, glitch_mode=glitch_mode, esw_mode=esw_mode)
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert r[key] == pytest.approx(b[key], rel=1e-11, abs=1e-22), key
    np.testing.assert_array_equal(r["glcount"], b["glcount"])
    np.testing.assert_array_equal(r["is_glitch"].astype(np.int64), b["is_glitch"])
    assert b["glcount"].sum() > 0


def test_brute_force_ties_are_exercised():
    # the quantised workloads above must contain cross-pin ties, else the tie rule is unpinned
    w = _tiny_random(3, 0.125, k_mode=2)
    pb = pin_base(w)
    ties = 0
    for g in range(len(w.cell_id)):
        k = int(w.n_inputs[w.cell_id[g]])
        times = [set(w.t_ns[int(w.pin_off[pb[g] + q]):int(w.pin_off[pb[g] + q + 1])].tolist()) for q in range(k)]
        for a in range(k):
            for b in range(a + 1, k):
                ties += len(times[a] & times[b])
    assert ties > 0


def test_gate_order_invariance():
    w = synth.generate(1)
    r = oracle.run(w)
    perm = np.random.default_rng(0).permutation(len(w.cell_id))
    pb = pin_base(w)
    t, s, v, po = [], [], [], [0]
    for g in perm:
        a, b = int(w.pin_off[pb[g]]), int(w.pin_off[pb[g + 1]])
        for p in range(int(pb[g]), int(pb[g + 1])):
            n = int(w.pin_off[p + 1] - w.pin_off[p])
            po.append(po[-1] + n)
        t.append(w.t_ns[a:b]); s.append(w.slew_ps[a:b]); v.append(w.value[a:b])
    import copy
    w2 = copy.copy(w)
    w2.cell_id, w2.load_ff = w.cell_id[perm], w.load_ff[perm]
    w2.init_in, w2.init_out = w.init_in[perm], w.init_out[perm]
    w2.pin_off = np.asarray(po, np.uint64)
    w2.t_ns, w2.slew_ps, w2.value = np.concatenate(t), np.concatenate(s), np.concatenate(v)
    r2 = oracle.run(w2)
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert r[key] == pytest.approx(r2[key], rel=1e-13)
    np.testing.assert_allclose(r["waveform"], r2["waveform"], rtol=1e-12)
    np.testing.assert_array_equal(r["evcount"], r2["evcount"])


def test_sampled_cycles_match_full_waveform():
    w = synth.generate(2)
    full = oracle.run(w, threads=4)
    cyc = np.array([0, 3, 17, 500, 998, 999, 250], np.uint32)
    smp = oracle.run(w, threads=4, wave="sample", sample_cycles=cyc)
    np.testing.assert_allclose(smp["waveform"], full["waveform"][cyc], rtol=1e-12)
    none = oracle.run(w, threads=4, wave="none")
    for key in ("p_int", "p_sw", "p_gl", "p_leak"):
        assert none[key] == pytest.approx(full[key], rel=1e-13)
    np.testing.assert_array_equal(none["evcount"], full["evcount"])


def test_generator_range_matches_full_slice():
    w = synth.generate(2)
    g0, g1 = 1234, 5678
    r = synth.generate_range(2, g0, g1)
    pb = pin_base(w)
    p0, p1 = int(pb[g0]), int(pb[g1])
    e0, e1 = int(w.pin_off[p0]), int(w.pin_off[p1])
    np.testing.assert_array_equal(r.pin_off, w.pin_off[p0:p1 + 1] - w.pin_off[p0])
    np.testing.assert_array_equal(r.t_ns, w.t_ns[e0:e1])
    np.testing.assert_array_equal(r.slew_ps, w.slew_ps[e0:e1])
    np.testing.assert_array_equal(r.value, w.value[e0:e1])
    np.testing.assert_array_equal(r.cell_id, w.cell_id[g0:g1])
    # the oracle on the block equals the oracle restricted to those gates (same events, same units)
    a = oracle.run(r, wave="none")
    b = oracle.run(w, wave="none", gate_range=(g0, g1))
    for key in ("e_int", "e_sw", "e_gl", "e_leak"):
        assert a[key] == pytest.approx(b[key], rel=1e-13)
