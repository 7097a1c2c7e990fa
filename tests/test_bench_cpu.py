"""Host logic of bench.py that needs no GPU: the full-size traffic derivation
from the small-case records (used only while the recorded kernel hash matches
the sources), the record file's consistency with its own derivation, and the
source hash's insensitivity to comments."""

import json

import pytest


@pytest.fixture(scope="module")
def bench():
    import bench as b
    return b


def test_traffic_derivation_and_hash_gate(bench, tmp_path, monkeypatch):
    h = bench.kernel_hash("full")
    rec = {"configs": {
        "1B/H8": {"family": "full", "kernel_hash": h, "tail_bytes": 60_000_000,
                  "output_bytes_per_token": 2560},
        "1B/H4": {"family": "full", "kernel_hash": "0" * 16, "tail_bytes": 1,
                  "output_bytes_per_token": 1}}}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    got = bench.measured_traffic("1B", 8, 7.72e9, 16384)
    assert got == pytest.approx(7.72e9 + 16384 * 2560 - 60_000_000)
    assert bench.measured_traffic("1B", 4, 7.72e9, 16384) is None      # stale hash
    assert bench.measured_traffic("1B", 16, 7.72e9, 16384) is None     # no record
    p.write_text("{not json")
    assert bench.measured_traffic("1B", 8, 7.72e9, 16384) is None      # unreadable


def test_committed_traffic_records_follow_their_own_derivation(bench):
    """Each committed record's tail is what its three small-case launches give:
    algorithmic bytes plus the output read per token, less the measured bytes,
    averaged; every measured launch stays within its algorithmic bytes plus that
    output (nothing re-read)."""
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)["configs"]
    assert rec
    for name, e in rec.items():
        T, ob = e["tokens"], e["output_bytes_per_token"]
        ls = e["launches"]
        assert len(ls) == 3, name
        tail = sum(l["algorithmic_bytes"] + T * ob - l["measured_bytes"] for l in ls) / 3
        assert abs(tail - e["tail_bytes"]) <= 1, name
        for l in ls:
            assert l["measured_bytes"] <= l["algorithmic_bytes"] + T * ob, name
        assert 20e6 < e["tail_bytes"] < 129e6, name   # below the 129 MB L2


def test_kernel_hash_ignores_comments(bench):
    code = "int a; // note\n/* block\n comment */\nint b;\n\n"
    assert bench._code_only(code) == bench._code_only("int a;\nint b;")
    assert bench._code_only("int a;") != bench._code_only("int b;")
