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


def test_flat_extras_are_scalars_named_for_their_leg():
    """The extra legs' summaries go into the JSON line's roofline object, where a parser
    that keeps only scalar fields must still find them: every value is a number."""
    link = {"h2d": 211.6, "d2h": 193.7, "bidir": 343.1}
    seq = {"store": {"gbs": 193.0, "frac": 0.996}, "load": {"gbs": 211.0, "frac": 0.997}}
    few = {k: {"gbs": 200.0, "frac": 0.95, "cfg": {"sm_cap": 4}}
           for k in ("load_bulk", "store_bulk", "load_segment", "store_segment")}
    mla = {"p1": {"store_frac": 0.96, "load_frac": 0.99},
           "p16": {"store_frac": 0.99, "load_frac": 0.99}}
    qwen = {"bound_ms": 51.0, "exchange_one_launch": {"frac_of_bound": 0.978},
            "two_streams": {"frac_of_bound": 0.93},
            "two_streams_store_16sm": {"frac_of_bound": 0.92},
            "two_streams_store_6sm": {"frac_of_bound": 0.977},
            "two_partitions": {"unavailable": "no green contexts"}}
    leg = {"load_overlap_gbs": 200.0, "gemm_slowdown_pct": 3.5, "e2e_vs_model": 1.02}
    l70 = {"bulk_6sm": leg, "bulk_5sm": leg, "bulk_4sm": leg, "segment_16sm": leg,
           "partition_16sm": {"unavailable": "no green contexts"}}
    evict = {"store_under_decode_gbs": 42.4, "decode_slowdown_pct": 0.8}
    f = bench.flat_extras(seq, few, mla, qwen, l70, evict, link)
    assert f and all(isinstance(v, (int, float)) for v in f.values())
    assert f["store_frac"] == 0.996 and f["load_frac"] == 0.997
    assert f["sm4_load_bulk_frac"] == 0.95 and f["cfg5_mla_p1_store_frac"] == 0.96
    assert f["cfg4_exchange_frac_of_bound"] == 0.978
    assert f["cfg4_two_streams_store_6sm_frac_of_bound"] == 0.977
    assert "cfg4_two_partitions_frac_of_bound" not in f  # an unavailable leg is left out
    assert f["cfg3_bulk_5sm_load_overlap_frac"] == round(200.0 / 211.6, 4)
    assert "cfg3_partition_16sm_gemm_slowdown_pct" not in f
    assert f["eviction_1sm_decode_slowdown_pct"] == 0.8
    # Without the extra legs only the per-direction figures remain.
    assert set(bench.flat_extras(seq, None, None, None, None, None, link)) == {
        "store_gbs", "store_frac", "load_gbs", "load_frac"}
