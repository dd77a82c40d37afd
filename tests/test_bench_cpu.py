"""bench.py's host-side choices, on the CPU: how many weight copies a timed
loop rotates through (enough to beat the L2, a divisor of both graph
lengths) and which workload --workload selects."""
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
