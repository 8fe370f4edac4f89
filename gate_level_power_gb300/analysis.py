"""Post-processing of the per-gate power a run returns (host-side analysis).

These helpers work on the ``gate_power`` / ``cell_power`` arrays that
``PowerAnalyzer.run`` returns; they are not part of the power computation,
which runs entirely in libpa.so's kernels, and they are kept out of the
binding module, which only marshals arguments. They give the spatial measures
of the paper's accuracy evaluation ("GPU-Accelerated Gate-Level Time-Based
Power Analysis via Event-Density-Aware Partitioning and Kernel Fusion",
Section 4, Fig. 10 and Table 3): hotspot lists, hotspot overlap@k and
Kendall's tau between two gate rankings.
"""
from __future__ import annotations

import numpy as np


def hotspots(power, frac: float = 0.01, component=None) -> np.ndarray:
    """Indices of the highest-power rows of a per-gate or per-cell power array
    ([n, 4] W: internal, switching, glitch, leakage), highest first: the top
    ``frac`` of the rows (at least one when there are any). ``component`` (0..3)
    ranks one column instead of the total. This is the hotspot list of the
    paper's spatial accuracy study (overlap@1%, Table 3)."""
    p = np.asarray(power, dtype=np.float64).reshape(-1, 4)
    v = p.sum(axis=1) if component is None else p[:, int(component)]
    n = max(1, int(np.ceil(frac * len(v)))) if len(v) else 0
    return np.argsort(-v, kind="stable")[:n]


def hotspot_overlap(a, b, frac: float = 0.01, component=None) -> float:
    """The fraction of the top-``frac`` hotspots of power array ``a`` that are
    also among the top-``frac`` hotspots of ``b`` (the paper's overlap@1%)."""
    ha, hb = hotspots(a, frac, component), hotspots(b, frac, component)
    return float(len(np.intersect1d(ha, hb))) / max(1, len(ha))


def rank_correlation(a, b, component=None) -> float:
    """Kendall's tau-b between the power rankings of two per-gate (or per-cell)
    power arrays (the paper's Fig. 10 compares gate rankings this way)."""
    from scipy.stats import kendalltau
    pa = np.asarray(a, dtype=np.float64).reshape(-1, 4)
    pb = np.asarray(b, dtype=np.float64).reshape(-1, 4)
    va = pa.sum(axis=1) if component is None else pa[:, int(component)]
    vb = pb.sum(axis=1) if component is None else pb[:, int(component)]
    return float(kendalltau(va, vb).statistic)
