"""CPU checks of bench.py's host-side helpers: the algorithmic byte count, the
traffic figure read from the committed ncu summaries (only for the kernel
source it was captured on), the generator overrides and the workload names."""
import os

import numpy as np

import bench
import synth


def test_algorithmic_bytes_counts_each_input_once():
    w = synth.generate(1)
    pins = int(w.n_pins)
    expect = 8 * w.n_events + 8 * (pins + 1) + 9 * w.n_gates + 12 * w.n_cycles + 4 * len(w.lut) + 4 * len(w.leak)
    assert bench.algorithmic_bytes(w) == expect
    # 8 bytes per event dominate the large workloads
    assert expect > 8 * w.n_events


def test_traffic_is_read_only_for_the_captured_source(monkeypatch, tmp_path):
    d = tmp_path / "profiles"
    d.mkdir()
    (d / "k.md").write_text("text\ntraffic_bytes_per_launch k_band config4: 1.5e10 source: abcdef0123456789\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "abcdef0123456789")
    assert bench.ncu_traffic("k_band", 4) == 1.5e10
    assert bench.ncu_traffic("k_band", 3) is None
    assert bench.ncu_traffic("k_fused", 4) is None
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "0000000000000000")
    assert bench.ncu_traffic("k_band", 4) is None


def test_committed_profile_names_a_traffic_figure():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "profiles", "k_band__config4_shape_200M_events.md")).read()
    assert "traffic_bytes_per_launch k_band config4:" in text


def test_source_digest_is_stable_and_short():
    a, b = bench.kernel_source_digest(), bench.kernel_source_digest()
    assert a == b and len(a) == 16 and all(ch in "0123456789abcdef" for ch in a)


def test_synth_overrides_and_workload_names():
    assert bench.synth_overrides(["n_gates=1000000", "n_events=200000000", "toggles=4"]) == {
        "n_gates": 1000000, "n_events": 200000000, "toggles": 4}
    assert bench.synth_overrides(["t_clk_ns=0.8", "zipf_s=1e0"]) == {"t_clk_ns": 0.8, "zipf_s": 1.0}
    cfg = synth.make_cfg(4, 0)
    G, _, E = synth.sizes(4, 0)
    wc = bench.workload_config(4, G, E, cfg)
    assert wc["workload"].startswith("config 4: very large skewed")
    assert wc["events"] == 1_000_000_000 and wc["cycles"] == 100_000 and "larger than L2" in wc["l2"]
    assert isinstance(np.float64(wc["t_clk_ns"]), np.floating)
