"""Host-side pieces of bench.py that need no GPU: the comment-insensitive source hash that
gates the recorded ncu traffic, and the traffic lookup itself."""
import os

import pytest

pytest.importorskip("torch")

import bench  # noqa: E402


def test_code_only_drops_comments_and_layout_but_keeps_strings():
    text = 'a = 1;   // note\n\n  b = "x // y /* z */";  /* block\n comment */ c;\n'
    assert bench._code_only(text) == 'a = 1;\nb = "x // y /* z */"; c;'
    # A comment or indentation edit leaves the code unchanged; a code edit does not.
    assert bench._code_only("x = 1; /* one */") == bench._code_only("  x = 1;  // two")
    assert bench._code_only("x = 1;") != bench._code_only("x = 2;")


def _fake_tree(root, kernels, internal, traffic_lines):
    csrc = root / "paged_kv_gather_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "kvx_kernels.cuh").write_text(kernels)
    (csrc / "kvx_internal.h").write_text(internal)
    (root / "profiles").mkdir()
    (root / "profiles" / "traffic.txt").write_text("\n".join(traffic_lines) + "\n")


def test_traffic_is_reported_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _fake_tree(tmp_path, "int k = 1; // kernels\n", "int i = 2;\n", ["# header"])
    sha = bench.source_sha()
    (tmp_path / "profiles" / "traffic.txt").write_text(
        f"kernel=roundtrip workload=llama8b source_sha={sha} dram_bytes_per_launch=800\n"
        f"kernel=exchange workload=llama8b source_sha={sha} dram_bytes_per_launch=1600\n")
    assert bench.recorded_traffic("roundtrip", "llama8b") == 800
    assert bench.recorded_traffic("exchange", "llama8b", groups=16) == 100
    assert bench.recorded_traffic("store", "llama8b") is None
    # A comment edit keeps the record; a code edit retires it.
    kernels = tmp_path / "paged_kv_gather_gb300" / "csrc" / "kvx_kernels.cuh"
    kernels.write_text("int k = 1;   /* reworded comment */\n")
    assert bench.recorded_traffic("roundtrip", "llama8b") == 800
    kernels.write_text("int k = 3;\n")
    assert bench.recorded_traffic("roundtrip", "llama8b") is None
    os.remove(tmp_path / "profiles" / "traffic.txt")
    assert bench.recorded_traffic("roundtrip", "llama8b") is None


def test_committed_traffic_records_name_a_source_hash():
    path = os.path.join(os.path.dirname(os.path.dirname(__file__)), "profiles", "traffic.txt")
    kernels = set()
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        f = dict(x.split("=", 1) for x in line.split())
        assert len(f["source_sha"]) == 16 and int(f["dram_bytes_per_launch"]) > 0
        kernels.add(f["kernel"])
    assert {"store", "load", "transform_gather", "transform_scatter", "roundtrip"} <= kernels
