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
    for kernel, entry in t["kernels"].items():
        name, value = next(iter(entry["bytes_per_launch"].items()))
        monkeypatch.setattr(bench, "kernel_source_hash", lambda k=kernel, e=entry: e["sha"])
        assert bench.main_kernel_traffic(name, kernel=kernel) == value
        # the counters belong to the default instance, not the deterministic one
        assert bench.main_kernel_traffic(name, deterministic=True, kernel=kernel) is None
        assert bench.main_kernel_traffic("no_such_workload", kernel=kernel) is None
        # sources changed since the capture: no figure
        monkeypatch.setattr(bench, "kernel_source_hash", lambda k=kernel: "0" * 16)
        assert bench.main_kernel_traffic(name, kernel=kernel) is None


def test_each_workload_names_the_kernel_the_library_runs():
    from flashattention_backward_preprocess_gb300.inputs import WORKLOADS
    assert bench.main_kernel_family(WORKLOADS["bf16_b4_h32_kv8_s2048_d128_causal"]) == "bwd_sm103_kernel"
    assert bench.main_kernel_family(WORKLOADS["bf16_b1_h16_kv4_s4096_d256_causal"]) == "bwd_d256_kernel"
    assert bench.main_kernel_family(WORKLOADS["fp32_b2_h8_kv2_s2048_d128_causal"]) == "bwd_simt_kernel"
