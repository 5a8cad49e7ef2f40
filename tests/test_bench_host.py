"""Host logic of bench.py that decides what the JSON line claims: the DRAM traffic of a profiled kernel is
reported only while the kernel's source files hash to the ones the ncu capture was taken on."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _record(tmp_path, src_text, recorded_text, nbytes=12345):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text(src_text)
    h = hashlib.sha256(recorded_text.encode()).hexdigest()[:16]
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# kernel, sources, sha256[:16], bytes per launch, summary\n"
        f"my_kernel k.cu {h} {nbytes} my_kernel.md\n")


def test_traffic_reported_while_sources_match(tmp_path, monkeypatch):
    _record(tmp_path, "kernel v1", "kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("my_kernel") == 12345
    assert bench.profiled_traffic("other_kernel") is None


def test_traffic_withheld_once_sources_changed(tmp_path, monkeypatch):
    _record(tmp_path, "kernel v2", "kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("my_kernel") is None


def test_committed_record_names_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.txt")) as f:
        for line in f:
            fields = line.split()
            if not fields or fields[0].startswith("#"):
                continue
            assert len(fields) == 5, line
            for src in fields[1].split(","):
                assert os.path.exists(os.path.join(ROOT, src)), src
            assert os.path.exists(os.path.join(ROOT, "profiles", fields[4])), fields[4]
            assert int(fields[3]) > 0
