"""Pins for the partition oracle (oracle/partition.py): the paper's per-gate
cycle partition (event-density-aware, Fig. 5) and the globally fixed one it is
compared with (Figs. 19 and 20). Checked against the limits and the additive
thread-count approximation the text derives, closed forms, and a brute-force
walk over every event. CPU only."""
import numpy as np
import pytest

import synth
from oracle import partition as P


@pytest.mark.parametrize("N,floor", [(1000, 1), (1000, 4), (100000, 8), (64, 64)])
def test_zero_event_gate_gets_the_parallelism_floor(N, floor):
    # sparse limit: with no events the thread count is the floor itself
    n = P.cycles_per_thread([0], N, P.PART_DENSITY, n_evt_tgt=8, n_thr_floor=floor)
    assert int(P.threads_per_gate(n, N)[0]) == floor
    assert int(n[0]) == N // floor


@pytest.mark.parametrize("tgt,floor", [(8, 1), (8, 16), (4, 2), (16, 100)])
def test_gate_at_the_target_density_gets_one_cycle_per_thread(tgt, floor):
    N = 10000
    for rho in (tgt, 2 * tgt, 50 * tgt):  # at least n_evt,tgt events per cycle
        n = P.cycles_per_thread([rho * N], N, P.PART_DENSITY, n_evt_tgt=tgt, n_thr_floor=floor)
        assert int(n[0]) == 1 and int(P.threads_per_gate(n, N)[0]) == N


def test_additive_thread_count_approximation():
    # N_thr ~ N_evt / n_evt,tgt + N_thr,floor (exact up to the rounding of
    # n_cyc and the ceiling): |N_cyc / n - N_cyc / x| <= N_cyc / (2 n x)
    rng = np.random.default_rng(5)
    N, tgt = 100000, 8
    for floor in (1, 10, 1000):
        n_evt = np.concatenate([[0, 1, 7, 8, 100], rng.integers(0, 40 * N, 2000)])
        n = P.cycles_per_thread(n_evt, N, P.PART_DENSITY, n_evt_tgt=tgt, n_thr_floor=floor)
        nthr = P.threads_per_gate(n, N)
        approx = n_evt / tgt + floor  # N_cyc is a multiple of every floor used
        x = N / approx                 # the unrounded cycles per thread
        ok = x >= 1
        bound = N / (2 * n * x) + 1
        assert np.all(np.abs(nthr - approx)[ok] <= bound[ok])
        # past one cycle per thread the count saturates at N_cyc
        assert np.all(nthr[~ok] == N)
        # sparse regime within 3 %, dense regime likewise (rounding of n only)
        big = x >= 20
        assert np.all(np.abs(nthr[big] - approx[big]) <= 0.03 * approx[big] + 1)


def test_density_partition_gives_more_threads_to_denser_gates():
    N = 20000
    n_evt = np.arange(0, 400000, 997)
    nthr = P.threads_per_gate(P.cycles_per_thread(n_evt, N, P.PART_DENSITY, n_evt_tgt=8, n_thr_floor=3), N)
    assert np.all(np.diff(nthr) >= 0)
    assert nthr[0] == 3 and nthr[-1] > 1000


@pytest.mark.parametrize("N,fix", [(1000, 1), (1000, 8), (1000, 7), (10, 32)])
def test_fixed_partition_threads(N, fix):
    n = P.cycles_per_thread([0, 5, 10 ** 6], N, P.PART_FIXED, n_cyc_fix=fix)
    assert np.all(P.threads_per_gate(n, N) == -(-N // min(fix, N)))


def _tiny(seed, n_gates=8, n_cycles=23, n_events=300, t_clk=0.7, k_mode=1):
    return synth.custom(seed=seed, n_gates=n_gates, n_cells=4, k_mode=k_mode, n_slew=4, n_load=3,
                        n_cycles=n_cycles, t_clk_ns=t_clk, n_events=n_events, pair_frac=0.2, threads=1)


@pytest.mark.parametrize("seed,mode,tgt,floor,fix", [
    (1, P.PART_DENSITY, 8, 1, 1), (2, P.PART_DENSITY, 2, 3, 1), (3, P.PART_DENSITY, 8, 23, 1),
    (4, P.PART_FIXED, 8, 1, 1), (5, P.PART_FIXED, 8, 1, 4), (6, P.PART_FIXED, 8, 1, 50)])
def test_thread_event_counts_match_brute_force(seed, mode, tgt, floor, fix):
    w = _tiny(seed)
    got = P.thread_event_counts(w, mode, tgt, floor, fix)
    ref = P.thread_event_counts_brute(w, mode, tgt, floor, fix)
    np.testing.assert_array_equal(got, ref)
    assert int(got.sum()) == len(w.t_ns)


def test_nearest_rank_quantiles():
    c = np.arange(1, 101)
    assert [P.nearest_rank(c, q) for q in (50, 90, 99, 100)] == [50, 90, 99, 100]
    assert P.nearest_rank([0, 0, 0, 5], 50) == 0 and P.nearest_rank([0, 0, 0, 5], 90) == 5
    assert P.nearest_rank([], 90) == 0
    assert P.nearest_rank([7], 1) == 7


def test_stats_of_a_standard_config():
    w = synth.generate(1)
    s = P.stats(w, P.PART_DENSITY)
    n_evt = P.gate_event_counts(w)
    assert s["threads"] == int(P.threads_per_gate(P.cycles_per_thread(n_evt, w.n_cycles, P.PART_DENSITY),
                                                  w.n_cycles).sum())
    assert s["p50"] <= s["p90"] <= s["p99"] <= s["max"]
    f = P.stats(w, P.PART_FIXED, n_cyc_fix=1)
    assert f["threads"] == len(n_evt) * w.n_cycles
