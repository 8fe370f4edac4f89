"""GPU parity of the warp kernel's partition corners against the oracle:
heavy gates whose pins differ widely in event count (the piece cut times
come from the densest pin, the windows share events by remaining counts),
events packed into bursts of a few cycles (many events of a pin per cycle,
glitch chains across window edges), and cross-pin ties on a coarse time grid
(timestamp groups at window edges), each at the default tile knobs and at
tiny ones that force many pieces and windows. The same workloads on the CTA
kernel with per-event outputs check the per-event states too."""
import numpy as np
import pytest

import oracle
import synth
from tests.test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu

KNOBS = [(0, 0), (8, 8), (64, 16), (1, 1), (400, 48)]  # 400 + 48: the largest tiles of the warp kernel


@pytest.fixture(scope="module")
def glp():
    import gate_level_power_gb300 as glp
    glp.build()
    glp.load_library()
    return glp


def hand_made(seed, pin_counts, n_cycles, t_clk, time_of):
    """A workload of one gate per entry of pin_counts (events per pin, the
    output last; the gate takes a cell with that many inputs), library and
    loads from the generator, event times from time_of(rng, pin, n) (sorted
    and made strictly increasing in f32), slews random, values toggling."""
    base = synth.custom(seed=seed, n_gates=len(pin_counts), n_cells=16, k_mode=1, n_slew=7, n_load=7,
                        n_cycles=n_cycles, t_clk_ns=t_clk, n_events=0, threads=1)
    rng = np.random.default_rng(seed)
    cell_id = []
    for counts in pin_counts:
        k = len(counts) - 1
        cells = np.nonzero(base.n_inputs == k)[0]
        assert len(cells), k
        cell_id.append(int(cells[rng.integers(len(cells))]))
    base.cell_id = np.asarray(cell_id, np.uint32)
    base.init_in = np.asarray([rng.integers(0, 1 << (len(c) - 1)) for c in pin_counts], np.uint8)
    base.init_out = rng.integers(0, 2, len(pin_counts)).astype(np.uint8)
    t_end = np.float32(n_cycles * t_clk)
    pin_off, ts, ss, vs = [0], [], [], []
    for g, counts in enumerate(pin_counts):
        k = len(counts) - 1
        for p, n in enumerate(counts):
            t = np.sort(np.asarray(time_of(rng, p, n), np.float32))
            for i in range(1, len(t)):  # strictly increasing in f32
                if t[i] <= t[i - 1]:
                    t[i] = np.nextafter(t[i - 1], np.float32(np.inf))
            assert len(t) == 0 or t[-1] < t_end
            init = (int(base.init_in[g]) >> p) & 1 if p < k else int(base.init_out[g])
            v = (init ^ ((np.arange(len(t)) + 1) & 1)).astype(np.uint8)
            ts.append(t)
            ss.append(rng.uniform(8.0, 300.0, len(t)).astype(np.float32))
            vs.append(v)
            pin_off.append(pin_off[-1] + len(t))
    base.pin_off = np.asarray(pin_off, np.uint64)
    base.t_ns = np.concatenate(ts).astype(np.float32)
    base.slew_ps = np.concatenate(ss).astype(np.float32)
    base.value = np.concatenate(vs).astype(np.uint8)
    return base


def check_all(glp, w):
    o = oracle.run(w, debug=True)
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        ref = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, debug=True)  # the CTA kernel, per-event outputs
        assert_parity(ref, o)
        for tile, heavy in KNOBS:
            r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, tile_events=tile, heavy_events=heavy)
            assert r["path"] == glp.PA_PATH_WARP
            try:
                assert_parity(r, o, debug=False)
            except AssertionError as e:
                raise AssertionError(f"knobs {tile}/{heavy}: {e}") from None
            if heavy:
                assert r["n_heavy"] > 0


def test_uneven_pins(glp):
    # one dense input pin among sparse ones (and a gate with a silent input pin)
    span = 300 * 1.0
    uni = lambda rng, p, n: rng.uniform(0.0, span * 0.999, n)
    w = hand_made(51, [(40000, 7, 3, 2000), (5, 6000, 4000), (9000, 0, 11, 300), (3, 2, 1, 1, 2)], 300, 1.0, uni)
    check_all(glp, w)


def test_bursts_in_few_cycles(glp):
    # most events of the gate packed into three cycles: many events of a pin
    # per cycle (glitch chains), windows cut inside the burst
    def burst(rng, p, n):
        nb = int(0.9 * n)
        return np.concatenate([rng.uniform(10.0, 13.0, nb), rng.uniform(0.0, 99.9, n - nb)])
    w = hand_made(52, [(3000, 500, 1000), (800, 800, 800, 800, 400), (2500, 40)], 100, 1.0, burst)
    check_all(glp, w)


def test_cross_pin_ties_on_a_grid(glp):
    # times on a 0.125 ns grid: many events of different pins at the same
    # time, so timestamp groups meet the window edges
    def grid(rng, p, n):
        return 0.125 * rng.choice(799, n, replace=False)
    w = hand_made(53, [(600, 600, 600, 600, 500), (700, 650, 300), (500, 500, 500, 300)], 100, 1.0, grid)
    check_all(glp, w)


def test_non_power_of_two_clock_bursts(glp):
    # the same bursts at a 0.7 ns clock (each cycle index an IEEE division)
    def burst(rng, p, n):
        nb = int(0.8 * n)
        return np.concatenate([rng.uniform(7.0, 9.1, nb), rng.uniform(0.0, 69.9, n - nb)])
    w = hand_made(54, [(2000, 2000, 900), (100, 3000, 30, 1200)], 100, 0.7, burst)
    check_all(glp, w)


def test_tile_limit_selects_the_kernel(glp):
    # tile_events + heavy_events up to 448 run on the warp kernel, above it on
    # the CTA kernel; both at the same bar against the oracle
    w = synth.custom(seed=57, n_gates=3000, n_cells=16, k_mode=1, n_cycles=200, t_clk_ns=1.0,
                     n_events=400000, activity=1, zipf_s=1.1, pair_frac=0.1, threads=4)
    o = oracle.run(w, threads=4)
    with glp.PowerAnalyzer(0) as pa:
        pa.load_workload(w)
        for tile, heavy, path in ((400, 48, glp.PA_PATH_WARP), (400, 49, glp.PA_PATH_UNBANDED)):
            r = pa.run(w.vdd, w.t_clk_ns, w.n_cycles, tile_events=tile, heavy_events=heavy)
            assert r["path"] == path, (tile, heavy)
            assert_parity(r, o, debug=False)
