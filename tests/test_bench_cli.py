"""bench.py's workload table and the kernel it names for the roofline (CPU only)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from exact_attention_blackwell_gb300 import inputs  # noqa: E402


def test_every_sweep_point_is_a_workload():
    names = set(bench.SWEEP_NAMES)
    assert len(names) == 18
    for w in inputs.sweep():
        got = bench.workload(bench.sweep_name(w.d, w.N, w.causal))
        assert (got.B, got.H, got.Hkv, got.N, got.d, got.causal) == (w.B, w.H, w.Hkv, w.N, w.d, w.causal)
        assert got.B * got.N == 32768 and got.H == 16


@pytest.mark.parametrize("name", ["headline", "causal", "gqa", "varlen"])
def test_named_workloads_match_their_configs(name):
    w = bench.workload(name)
    shape = {"headline": (4, 16, 16, 8192, 128, False), "causal": (8, 16, 16, 4096, 128, True),
             "gqa": (1, 32, 8, 32768, 128, True)}.get(name)
    if shape is not None:
        assert (w.B, w.H, w.Hkv, w.N, w.d, w.causal) == shape


def test_committed_profile_summaries_carry_traffic_and_a_source_hash():
    # every summary bench.py may read names a traffic figure and the sources it was taken on
    prof = os.path.join(ROOT, "profiles")
    for f in os.listdir(prof):
        if not f.endswith(".md") or f.startswith("launches"):
            continue
        text = open(os.path.join(prof, f)).read()
        if "traffic_bytes_per_launch" in text:
            assert "source_sha:" in text, f
