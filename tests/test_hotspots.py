"""CPU checks of the per-gate power analysis helpers: hotspot lists, their
overlap (the paper's overlap@1%) and Kendall's tau between rankings."""
import numpy as np
import pytest

from gate_level_power_gb300 import analysis


def test_hotspots_rank_by_total_or_component():
    p = np.zeros((300, 4))
    p[:, 0] = np.arange(300)          # internal power rises with the index
    p[:, 2] = np.arange(300)[::-1]    # glitch power falls with it
    p[7, 3] = 1e6                     # one gate dominated by leakage
    assert analysis.hotspots(p, 0.01).tolist() == [7, 0, 1]
    assert analysis.hotspots(p, 0.01, component=0).tolist() == [299, 298, 297]
    assert analysis.hotspots(p, 0.01, component=2).tolist() == [0, 1, 2]
    assert len(analysis.hotspots(p[:5], 0.01)) == 1 and len(analysis.hotspots(np.zeros((0, 4)))) == 0


def test_overlap_and_rank_correlation():
    rng = np.random.default_rng(0)
    p = rng.random((1000, 4))
    assert analysis.hotspot_overlap(p, p) == 1.0
    assert analysis.rank_correlation(p, p) == pytest.approx(1.0)
    assert analysis.rank_correlation(p, -p) == pytest.approx(-1.0)
    q = p.copy()
    top = analysis.hotspots(p, 0.01)
    q[top] = 0.0                      # the top 1% of p drop out of q's top 1%
    assert analysis.hotspot_overlap(p, q) == 0.0
    assert 0.9 < analysis.rank_correlation(p, q) < 1.0
