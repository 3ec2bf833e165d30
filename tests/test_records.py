"""The committed measurement records stay consistent with the sources (CPU only): the gate/up
DRAM-traffic record that bench.py reports belongs to the current bf16 grouped-GEMM sources, and
every profile summary names the command that produced it."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_record_matches_the_gemm_sources():
    """A traffic figure is reported only while the kernel sources are the captured ones; a stale
    record makes the bench print null instead of an old kernel's bytes."""
    rec = json.load(open(os.path.join(ROOT, "profiles", "gate_up_traffic.json")))
    if rec["source_sha256_prefix"] != bench.gemm_source_sha():
        assert bench.measured_traffic("v4flash_T8192") is None
        return
    assert bench.measured_traffic("v4flash_T8192") is not None
    # the capture stays within the kernel's algorithmic bytes plus its intermediates (no wasted
    # re-reads of the weights)
    from routed_expert_swiglu_gb300 import workloads
    w = workloads.V4FLASH_T8192
    alg = bench.gate_up_bytes(w, w.E) + bench.gate_up_intermediate_bytes(w)
    assert 0.95 < rec["scaled_bytes_per_launch"]["v4flash_T8192"] / alg < 1.10


def test_profile_summaries_name_their_commands():
    d = os.path.join(ROOT, "profiles")
    for name in sorted(os.listdir(d)):
        if name.endswith(".md"):
            text = open(os.path.join(d, name)).read()
            assert "ncu " in text and "--clock-control none" in text, name
            assert "python bench.py" in text, name
