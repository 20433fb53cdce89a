"""The bench's host-side bookkeeping on CPU: the recorded DRAM traffic of the
dominant kernel is reported only while it still describes today's kernel."""
import json
import os
import shutil

import bench

SRC = os.path.join(bench.ROOT, "collective_communication_schedules_gb300", "csrc", "reduce.cu")


def _fake_root(tmp_path, source_text):
    """A repo tree with the committed traffic record and the given reduce.cu."""
    os.makedirs(tmp_path / "profiles")
    os.makedirs(tmp_path / "collective_communication_schedules_gb300" / "csrc")
    shutil.copy(os.path.join(bench.ROOT, "profiles", "traffic.json"), tmp_path / "profiles" / "traffic.json")
    (tmp_path / "collective_communication_schedules_gb300" / "csrc" / "reduce.cu").write_text(source_text)
    return str(tmp_path)


def _record():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)["fused_reduce_broadcast"]


def test_comment_edits_keep_the_record(tmp_path, monkeypatch):
    e = _record()
    text = open(SRC).read()
    edited = "// a new header line\n\n" + text.replace("\n", "  // trailing note\n", 3)
    monkeypatch.setattr(bench, "ROOT", _fake_root(tmp_path, edited))
    got = bench.recorded_traffic("fused_reduce_broadcast", e["k"], e["count"])
    want = e["bytes_per_launch"] if bench.hashlib.sha256(bench.source_code(text)).hexdigest()[:16] == \
        e["code_sha256_16"] else None
    assert got == want


def test_code_edits_drop_the_record(tmp_path, monkeypatch):
    e = _record()
    text = open(SRC).read() + "\nstatic int changed_code = 1;\n"
    monkeypatch.setattr(bench, "ROOT", _fake_root(tmp_path, text))
    assert bench.recorded_traffic("fused_reduce_broadcast", e["k"], e["count"]) is None


def test_other_workloads_get_no_record():
    e = _record()
    assert bench.recorded_traffic("fused_reduce_broadcast", e["k"] - 1, e["count"]) is None
    assert bench.recorded_traffic("fused_reduce_broadcast", e["k"], e["count"] // 2) is None
    assert bench.recorded_traffic("no_such_kernel", e["k"], e["count"]) is None


def test_record_agrees_with_its_own_counters():
    e = _record()
    assert e["bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
    # within a few per cent of the algorithmic 2kS of one fused allreduce launch
    algorithmic = 2 * e["k"] * e["count"] * 2
    assert abs(e["bytes_per_launch"] / algorithmic - 1) < 0.05
