"""bench.py's recorded DRAM traffic: every record points at a committed ncu summary that carries the same
kernel-source hash, and a record goes null (not stale) once the kernel code it was taken on changes."""
import json
import os
import re
import shutil

import bench

ROOT = os.path.join(os.path.dirname(__file__), "..")


def test_every_traffic_record_names_a_profile_with_its_source_hash():
    rec = json.load(open(os.path.join(ROOT, "profiles", "engine_traffic.json")))
    assert set(rec) >= {"decode", "prefill", "stacked_qkv", "stacked_gate_up", "stacked_down", "moe"}
    for name, entry in rec.items():
        assert entry["dram_bytes_per_launch"] > 0, name
        m = re.search(r"profiles/[A-Za-z0-9_.]+\.md", entry["source"])
        assert m, name
        text = open(os.path.join(ROOT, m.group(0))).read()
        assert entry["engine_sha"] in text, (name, m.group(0))


def test_traffic_survives_comment_edits_and_goes_null_on_code_edits(tmp_path, monkeypatch):
    csrc = tmp_path / "segmented_rank_gemm_lora_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in set(bench.ENGINE_SOURCES) | set(bench.LINEAR_SOURCES) | set(bench.EMBED_SOURCES):
        shutil.copy(os.path.join(ROOT, "segmented_rank_gemm_lora_gb300", "csrc", name), csrc / name)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.engine_source_sha()
    (tmp_path / "profiles" / "engine_traffic.json").write_text(json.dumps(
        {"stacked_gate_up": {"engine_sha": sha, "dram_bytes_per_launch": 123, "source": "test"}}))
    assert bench.recorded_traffic("stacked_gate_up") == 123
    stream = csrc / "stream.cu"
    stream.write_text(stream.read_text() + "\n// a comment only\n/* and a block comment */\n")
    assert bench.recorded_traffic("stacked_gate_up") == 123
    stream.write_text(stream.read_text() + "\nnamespace lora { constexpr int kProbe = 1; }\n")
    assert bench.recorded_traffic("stacked_gate_up") is None
    # the other kernels' records hash their own sources
    assert bench.engine_source_sha(bench.LINEAR_SOURCES) != bench.engine_source_sha()
    assert bench.recorded_traffic("linear_prefill") is None   # no record for it in this file
