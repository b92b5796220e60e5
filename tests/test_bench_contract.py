"""bench.py's contract on the host (no GPU): the reference arm (the CPU
oracle) prints one JSON line with exactly the K and W it was given and the
same `config` as the GPU arm, and the region helper times exactly the work
it is handed."""
import json
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _FakeLayers:
    """Stands in for the oracle's layer copies: counts steps, no arithmetic."""
    weight_bytes = 1_000_000

    def __init__(self):
        self.calls = []
        self.copies = [None] * 8

    def step(self, i):
        self.calls.append(i)


def test_reference_arm_line_matches_the_gpu_arms_contract(capsys, monkeypatch):
    fake = _FakeLayers()
    monkeypatch.setattr(bench, "OracleLayers", lambda: fake)
    monkeypatch.setattr(bench, "REF_MIN_SECONDS", 0.0)
    monkeypatch.setattr(bench, "REF_MAX_SECONDS", 5.0)
    bench.run_reference(types.SimpleNamespace(steps=20, warmup=5), world=1, rank=0)
    line = json.loads(capsys.readouterr().out)
    assert line["impl"] == "reference"
    assert line["steps"] == 20 and line["warmup"] == 5
    assert line["config"] == bench.headline_config(1)
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # W untimed steps, then regions of exactly K consecutive steps
    regions = line["timing"]["regions"]
    assert fake.calls == list(range(5 + 20 * regions))


def test_headline_config_names_the_workload_and_l2_rule():
    cfg = bench.headline_config(2)
    assert cfg["weight_bytes_per_step"] == 63_191_040
    assert "larger than L2" in cfg["l2"]
    assert cfg["parallelism"] == "replicas x2"
    assert len(cfg["matrices"]) == 7
