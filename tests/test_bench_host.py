"""Host-side logic of bench.py that needs no GPU: the ncu traffic figure it reports."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _traffic_json():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


def test_traffic_reported_only_for_the_captured_kernel(monkeypatch):
    t = _traffic_json()
    name = "bf16_b4_h32_kv8_s2048_d128_causal"
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: t["kernel_sha"])
    assert bench.main_kernel_traffic(name) == t["bytes_per_launch"][name]
    # the counters belong to the default instance, not the deterministic one
    assert bench.main_kernel_traffic(name, deterministic=True) is None
    assert bench.main_kernel_traffic("no_such_workload") is None
    # sources changed since the capture: no figure
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.main_kernel_traffic(name) is None

