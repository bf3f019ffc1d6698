"""Host logic of the measurement (no GPU): the DRAM traffic a bench line reports comes
from a committed ncu summary only while the summarised kernel's sources are unchanged,
and the roofline peaks come from the measured-peaks file, else the stated fallback."""
import json
import os

import pytest

import bench


@pytest.fixture
def tree(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text("// kernel v1\n")
    (tmp_path / "h.cuh").write_text("// helper\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def write_summary(tree, name, traffic, sha):
    (tree / "profiles" / name).write_text(
        f"# summary\n\ntraffic_bytes_per_launch: {traffic}\nsource_sha256: {sha}\n")


def test_traffic_is_read_while_the_sources_match(tree):
    srcs = ["k.cu", "h.cuh"]
    write_summary(tree, "k.md", 123456, bench.source_sha(srcs))
    assert bench.profiled_traffic("k.md", srcs) == 123456


def test_traffic_goes_null_once_a_source_changes(tree):
    srcs = ["k.cu", "h.cuh"]
    write_summary(tree, "k.md", 123456, bench.source_sha(srcs))
    (tree / "h.cuh").write_text("// helper, edited\n")
    assert bench.profiled_traffic("k.md", srcs) is None


def test_traffic_is_null_without_a_summary_or_its_lines(tree):
    srcs = ["k.cu"]
    assert bench.profiled_traffic("missing.md", srcs) is None
    (tree / "profiles" / "bare.md").write_text("# no counters here\n")
    assert bench.profiled_traffic("bare.md", srcs) is None


def test_source_hash_depends_on_order_and_content(tree):
    a = bench.source_sha(["k.cu", "h.cuh"])
    assert a == bench.source_sha(["k.cu", "h.cuh"])
    assert a != bench.source_sha(["h.cuh", "k.cu"])
    assert len(a) == 16 and int(a, 16) >= 0


def test_measured_peaks_file_else_fallback(tree):
    assert bench.measured_peaks() == (6800.0, 1900.0, 1700.0, "fallback")
    (tree / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6766.4, "bf16_tflops": 1943.4, "bf16_tflops_sustained": 1730.1}))
    assert bench.measured_peaks() == (6766.4, 1943.4, 1730.1, "measured")
    (tree / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000, "bf16_tflops": 2000}))
    # no sustained figure: the burst one stands in for it
    assert bench.measured_peaks() == (7000.0, 2000.0, 2000.0, "measured")


def test_committed_summaries_carry_counters_for_the_current_sources():
    # every bench workload that reports traffic names a committed summary with the two
    # lines the lookup reads (whether the hash matches depends on the tree's history)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for name in ("attention_llama8b_decode.md", "prefill_tc_varlen_mixed.md",
                 "sparse_partials_block_sparse.md", "sparse_tc16_block_sparse_f16.md"):
        text = open(os.path.join(root, "profiles", name)).read()
        assert "traffic_bytes_per_launch:" in text and "source_sha256:" in text, name
        assert "ncu " in text and "--clock-control none" in text, name
