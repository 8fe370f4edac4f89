"""Randomised GPU parity: small seeded workloads drawn over the generator's
knobs (gates, cells and input counts, table sizes, clock, cycles, event count,
pulse pairs, time quantum for ties, bursts, skew), each run through every path
-- the unbanded kernel, the banded kernel at a random band size (per-event and
timed variants) and the paper's window partition -- against the fp64 oracle at
the usual bar (states, LUT intervals, glitch flags and counts bit-exact; totals
within 1e-5; bins within 1e-4 of the peak)."""
import numpy as np
import pytest

import oracle
import synth
from tests.test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu

SEEDS = list(range(32))


@pytest.fixture(scope="module")
def glp():
    import gate_level_power_gb300 as glp
    glp.build()
    glp.load_library()
    return glp


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    n_gates = int(rng.integers(5, 300))
    n_cycles = int(rng.integers(3, 400))
    kw = dict(seed=seed, n_gates=n_gates, n_cells=int(rng.integers(2, 17)), k_mode=int(rng.integers(0, 3)),
              n_slew=int(rng.integers(2, 9)), n_load=int(rng.integers(2, 9)), n_cycles=n_cycles,
              t_clk_ns=float(rng.choice([1.0, 0.5, 0.7, 1.3, 2.0])),
              n_events=int(rng.integers(0, 40 * n_gates + 1)), pair_frac=float(rng.choice([0.0, 0.1, 0.4])),
              quantum_ns=float(rng.choice([0.0, 0.0, 0.25, 1 / 16, 0.05])), threads=2)
    if rng.random() < 0.3:
        kw.update(burst_frac=0.8, burst_width=int(rng.integers(1, 4)), burst_cover=0.1)
    band = int(rng.choice([0, 1, 2, 8, 64]))
    return kw, band


@pytest.mark.parametrize("seed", SEEDS)
def test_random_workload_on_every_path(glp, seed):
    kw, band = draw(seed)
    w = synth.custom(**kw)
    o = oracle.run(w, debug=True)
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        runs = {"unbanded": pa.run(w.vdd, w.t_clk_ns, w.n_cycles, debug=True),
                "unbanded timed": pa.run(w.vdd, w.t_clk_ns, w.n_cycles),
                "unbanded timed, small tiles": pa.run(w.vdd, w.t_clk_ns, w.n_cycles, tile_events=16,
                                                      heavy_events=8),
                "window density": pa.run(w.vdd, w.t_clk_ns, w.n_cycles, debug=True, partition="density"),
                "window fixed": pa.run(w.vdd, w.t_clk_ns, w.n_cycles, partition="fixed", n_cyc_fix=3)}
        pa.build_bands(w.t_clk_ns, band)
        runs["banded"] = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, debug=True)
        runs["banded timed"] = pa.run(w.vdd, w.t_clk_ns, w.n_cycles)
    for name, r in runs.items():
        try:
            assert_parity(r, o, debug="state_pre" in r)
        except AssertionError as e:
            raise AssertionError(f"{name} ({kw}, band {band}): {e}") from None
