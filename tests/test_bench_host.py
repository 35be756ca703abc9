"""Host-side logic of bench.py (no GPU): the algorithmic work per unit that the rooflines divide
by, and the gating of recorded DRAM traffic by the hashes of the kernel sources it was measured
on."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_flops_per_pair_counts():
    # moments: the logit (2d) and omega, sum w k, the upper triangle of sum w k k^T (2 each)
    assert bench.moments_flops_per_pair(64) == 128 + 2 * (1 + 64 + 64 * 65 // 2) == 4418
    # the contraction alone: omega, sum w k, the upper triangle of sum w k k^T
    assert bench.contraction_flops_per_pair(64) == 2 * (1 + 64 + 64 * 65 // 2) == 4290
    # executed on the tensor cores: hi and lo over 5 passes of 448 feature columns; the weight
    # sweeps run Q K^T twice
    assert bench.tc_executed_flops_per_pair(64) == 2 * 2 * 5 * 448 == 8960
    assert bench.tc_weights_executed_flops_per_pair(64) == 2 * 2 * 64
    # Parallax forward: q.k, r.k, P1 V, P2 V
    assert bench.parallax_flops_per_pair(64, 64) == 512
    # Parallax backward: the record pass (4d + 4dv), then q.k, r.k, dO.v once, dq, dr, dk, dv
    alg, exe = bench.parallax_bwd_flops_per_pair(64, 64)
    assert alg == 16 * 64 + 8 * 64 == 1536
    assert exe == 20 * 64 + 10 * 64


def test_causal_pairs_of_the_headline_workload():
    from local_linear_attention_gb300 import workloads as W
    w = W.WORKLOADS[3]
    assert bench.causal_pairs(w) == w.B * w.H * w.T * (w.T + 1) // 2 == 268500992


@pytest.fixture
def traffic_file(tmp_path, monkeypatch):
    """A traffic record in a scratch profiles/ directory, with controllable source hashes."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    shas = {"a.cu": "aaaa", "b.cu": "bbbb"}
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda name: shas[name])
    rec = {"a.cu": {"source_sha": "aaaa", "dram_bytes_per_launch": 123},
           "b.cu": {"source_sha": "bbbb", "depends": {"a.cu": "aaaa"},
                    "dram_bytes_per_launch": 456}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    return shas


def test_recorded_traffic_current_sources(traffic_file):
    assert bench.recorded_traffic("a.cu") == 123
    assert bench.recorded_traffic("b.cu") == 456
    assert bench.recorded_traffic("c.cu") is None  # no record


def test_recorded_traffic_is_dropped_when_a_source_changes(traffic_file):
    traffic_file["a.cu"] = "changed"
    assert bench.recorded_traffic("a.cu") is None
    # b.cu itself is unchanged, but its step also launches a kernel of a.cu
    assert bench.recorded_traffic("b.cu") is None


def test_committed_traffic_records_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    csrc = os.path.join(ROOT, "local_linear_attention_gb300", "csrc")
    for name, ent in rec.items():
        assert os.path.exists(os.path.join(csrc, name)), name
        assert ent["dram_bytes_per_launch"] > 0
        for dep in ent.get("depends", {}):
            assert os.path.exists(os.path.join(csrc, dep)), dep
