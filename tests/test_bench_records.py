"""bench.py's measurement helpers (CPU): the committed ncu traffic record is
used only while the kernel's code is the code it was captured from (comments
and whitespace aside), and per-launch times are summarised as mean, best and
median."""
import json
import os
import shutil

import bench


def _tree(tmp_path, src_text):
    csrc = tmp_path / "collective_transport_plane_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(src_text)
    (tmp_path / "profiles").mkdir()
    return str(tmp_path)


def _record(root, h, traffic=12345):
    rec = {"sources": ["k.cu"], "kernel_source_hash": h, "traffic_bytes_per_launch": traffic}
    with open(os.path.join(root, "profiles", "rec.json"), "w") as f:
        json.dump(rec, f)


def test_traffic_record_follows_the_code(tmp_path):
    root = _tree(tmp_path, "int f() { return 1; }  // one\n")
    h = bench.kernel_source_hash(["k.cu"], root)
    _record(root, h)
    assert bench.profiled_traffic("rec", root) == 12345
    # comments and whitespace do not make the record stale
    (tmp_path / "collective_transport_plane_gb300" / "csrc" / "k.cu").write_text(
        "/* header */\nint f()  {\n  return 1;\n}\n")
    assert bench.profiled_traffic("rec", root) == 12345
    # a change of code does
    (tmp_path / "collective_transport_plane_gb300" / "csrc" / "k.cu").write_text("int f() { return 2; }\n")
    assert bench.profiled_traffic("rec", root) is None


def test_traffic_record_missing_or_unreadable(tmp_path):
    root = _tree(tmp_path, "int f();\n")
    assert bench.profiled_traffic("rec", root) is None
    with open(os.path.join(root, "profiles", "rec.json"), "w") as f:
        f.write("{not json")
    assert bench.profiled_traffic("rec", root) is None
    shutil.rmtree(os.path.join(root, "collective_transport_plane_gb300"))
    _record(root, "0" * 16)
    assert bench.profiled_traffic("rec", root) is None


def test_committed_records_name_their_sources():
    prof = os.path.join(bench.ROOT, "profiles")
    for name in os.listdir(prof):
        if not name.endswith(".json"):
            continue
        rec = json.load(open(os.path.join(prof, name)))
        assert rec["sources"] and rec["kernel_source_hash"] and rec["traffic_bytes_per_launch"] > 0, name
        for f in rec["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, "collective_transport_plane_gb300", "csrc", f)), (name, f)


def test_committed_records_match_their_summaries():
    # each machine-readable record sits beside the text summary of the same
    # capture, which names the same kernel source hash
    prof = os.path.join(bench.ROOT, "profiles")
    for name in os.listdir(prof):
        if not name.endswith(".json"):
            continue
        rec = json.load(open(os.path.join(prof, name)))
        md = os.path.join(prof, name[:-len(".json")] + ".md")
        assert os.path.exists(md), name
        assert rec["kernel_source_hash"] in open(md).read(), name


def test_time_stats():
    st = bench.time_stats([0.5, 0.4, 0.7, 0.45])
    assert st["ms_best"] == 0.4
    assert st["ms_median"] == 0.475
    assert abs(st["ms_mean"] - 0.5125) < 1e-12
