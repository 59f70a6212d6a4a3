"""The bench line's committed ncu figures (profiles/traffic.json): used only
for the bench mode they were captured in, and only while the kernel sources
they depend on are byte for byte those of the capture (CPU)."""
import hashlib
import json
import os
import shutil

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _copy_tree(tmp_path):
    """The record and the kernel sources it names, in a scratch root, the
    record's hash taken over those sources (so it is current there whether
    or not the committed one is)."""
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "bit_trellis_quantized_gb300" / "csrc"
    csrc.mkdir(parents=True)
    h = hashlib.sha256()
    for src in rec["sources"]:
        shutil.copy(os.path.join(ROOT, "bit_trellis_quantized_gb300", "csrc", src), csrc / src)
        h.update((csrc / src).read_bytes())
    rec["sources_sha256"] = h.hexdigest()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    return rec, csrc


def test_record_names_existing_sources_and_a_capture():
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for key in ("kernel", "mode", "dram_bytes_per_launch", "instructions_per_weight", "sources", "sources_sha256",
                "capture"):
        assert key in rec, key
    for src in rec["sources"]:
        assert os.path.exists(os.path.join(ROOT, "bit_trellis_quantized_gb300", "csrc", src)), src
    assert os.path.exists(os.path.join(ROOT, rec["capture"]))
    assert rec["dram_bytes_per_launch"] > 0 and rec["instructions_per_weight"] > 0


def test_record_used_only_in_its_mode_and_while_sources_match(tmp_path, monkeypatch):
    rec, csrc = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    mode = rec["mode"]
    other = "sequence" if mode != "sequence" else "blocks"
    assert bench.measured_traffic(mode) == rec["dram_bytes_per_launch"]
    assert bench.measured_instr_per_weight(mode) == rec["instructions_per_weight"]
    assert bench.measured_traffic(other) is None
    assert bench.measured_traffic(None) is None
    # any change to a source the record depends on retires it
    src = csrc / rec["sources"][-1]
    src.write_bytes(src.read_bytes() + b"\n// changed\n")
    assert bench.measured_traffic(mode) is None
    assert bench.measured_instr_per_weight(mode) is None


def test_missing_record_gives_none(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("blocks") is None
    assert bench.measured_instr_per_weight("blocks") is None
