"""bench.py's host-side choices, on the CPU: how many weight copies a timed
loop rotates through (enough to beat the L2, a divisor of both graph
lengths), which workload --workload selects, when the recorded ncu traffic
still describes the kernel (its key ignores comments and layout, not code),
where the roofline's peak comes from, and the single-process aggregate."""
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402
import synthetic  # noqa: E402


def test_weight_copies_beat_the_l2_and_divide_the_graphs():
    for wl in (synthetic.HEADLINE, synthetic.GRAPH_8192, synthetic.CHAIN_4096):
        c = bench.weight_copies(wl.weight_bytes)
        assert bench.GRAPH_STEPS % c == 0 and bench.E2E_GRAPH_STEPS % c == 0
        assert c * wl.weight_bytes > 2 * bench.L2_BYTES, (wl.name, c)
    # The two bandwidth workloads rotate more than 12 x the L2, so no call finds
    # another call's weight there (three copies of the headline weight left
    # 8-10 % of each call's bytes in L2).
    assert bench.weight_copies(synthetic.HEADLINE.weight_bytes) == 15
    assert bench.weight_copies(synthetic.GRAPH_8192.weight_bytes) == 30
    for wl in (synthetic.HEADLINE, synthetic.GRAPH_8192):
        c = bench.weight_copies(wl.weight_bytes)
        assert c * wl.weight_bytes >= bench.ROTATION_L2_MULTIPLE * bench.L2_BYTES
        assert "every call reads its weight from HBM" in bench.rotation_note(c, wl.weight_bytes)
    # A weight too small to outgrow the L2 gets the largest rotation.
    assert bench.weight_copies(synthetic.TINY.weight_bytes) == 30
    assert "latency" in bench.rotation_note(30, synthetic.TINY.weight_bytes)


def test_workload_selection():
    try:
        for name, attr in bench.WORKLOAD_CHOICES.items():
            bench._WORKLOAD = name
            assert bench.workload() is getattr(synthetic, attr)
        assert bench.parse_args([]).workload == "headline"
    finally:
        bench._WORKLOAD = "headline"


def _copy_kernel_sources(dst: Path, edit=None) -> None:
    for rel in bench.KERNEL_SOURCES:
        text = (ROOT / rel).read_text()
        out = dst / rel
        out.parent.mkdir(parents=True, exist_ok=True)
        out.write_text(edit(text) if edit else text)


def test_traffic_key_ignores_comments_and_layout_only(tmp_path, monkeypatch):
    """The recorded DRAM traffic stays valid across comment and whitespace
    edits of the kernel sources, and lapses with any change of their code."""
    assert list(bench._code_lines("a = 1;  // note\n\n   // only a comment\n  b();\n")) == \
        ["a = 1;", "  b();"]
    want = bench.kernel_source_hash()
    variants = {
        "comment": lambda t: t.replace("\n", "\n// an added comment line\n", 1),
        "layout": lambda t: t.replace(";\n", ";   \n\n", 3),
        "code": lambda t: t.replace("namespace mxfp8 {", "namespace mxfp8 {\nconstexpr int kProbe = 1;", 1),
    }
    got = {}
    for name, edit in variants.items():
        root = tmp_path / name
        _copy_kernel_sources(root, edit)
        monkeypatch.setattr(bench, "ROOT", root)
        got[name] = bench.kernel_source_hash()
    assert got["comment"] == want and got["layout"] == want
    assert got["code"] != want


def test_recorded_traffic_only_for_the_kernel_it_was_taken_on(tmp_path, monkeypatch):
    import json
    rec = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", rec)
    rec.write_text(json.dumps({"kernel_source_sha256_16": bench.kernel_source_hash(),
                               "dram_bytes_per_launch": 123}))
    assert bench.recorded_traffic() == 123
    monkeypatch.setattr(bench, "_WORKLOAD", "chain")  # taken on the headline workload only
    assert bench.recorded_traffic() is None
    monkeypatch.setattr(bench, "_WORKLOAD", "headline")
    rec.write_text(json.dumps({"kernel_source_sha256_16": "0" * 16, "dram_bytes_per_launch": 123}))
    assert bench.recorded_traffic() is None
    rec.write_text("not json")
    assert bench.recorded_traffic() is None


def test_peak_is_the_measured_copy_bandwidth_else_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6677.8, "bf16_tflops": 1900}')
    assert bench.measured_peak() == (6677.8, "measured")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"bf16_tflops": 1900}')
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")


def test_single_process_aggregate_is_the_identity():
    assert bench.aggregate(1.5, 42.0, group_initialised=False) == (1.5, 42.0)
