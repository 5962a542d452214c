"""The benchmark's recorded DRAM traffic and the committed ncu summaries (host-only checks)."""
import glob
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_record_is_keyed_by_the_kernel_source(monkeypatch, tmp_path):
    """roofline.traffic comes from profiles/traffic.txt only while the kernel source hash matches:
    a record under another hash, or for another workload, reads as None."""
    rec = tmp_path / "profiles"
    rec.mkdir()
    (rec / "traffic.txt").write_text("# comment\nabc123 square4096 23346176\nabc123 other 5\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_hash", lambda: "abc123")
    assert bench.recorded_traffic("square4096") == 23346176
    assert bench.recorded_traffic("lm_head") is None
    monkeypatch.setattr(bench, "kernel_hash", lambda: "def456")
    assert bench.recorded_traffic("square4096") is None


def test_kernel_hash_covers_the_kernel_source():
    h = bench.kernel_hash()
    assert re.fullmatch(r"[0-9a-f]{16}", h)
    assert h == bench.kernel_hash()


def test_every_profile_names_its_command_with_unlocked_clocks():
    """Each ncu summary gives the command that made it, and every ncu command there leaves the
    GPU clocks alone (--clock-control none)."""
    files = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
    assert files
    for f in files:
        text = open(f).read()
        blocks = re.findall(r"```\n(.*?)```", text, flags=re.S)  # the command blocks
        cmds = [line for blk in blocks for line in blk.splitlines() if line.lstrip().startswith("ncu ")]
        assert cmds, f"{os.path.basename(f)} names no ncu command"
        for c in cmds:
            assert "--clock-control none" in c, f"{os.path.basename(f)}: {c}"
