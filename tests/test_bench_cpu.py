"""Host-side arithmetic of bench.py on CPU: the roofline's algorithmic bytes and
useful FLOPs per launch (closed forms of the five workloads), and the rule that
a recorded ncu traffic figure is reported only for the kernel source it was
measured on."""
import json

import pytest

import bench
from conv2d_backward_implicit_gb300 import workloads


def test_algorithmic_bytes_closed_forms():
    # |grad_out| + |weight| (input dtype) + |grad_in| (float32), each once.
    want = {
        "resnet": 32 * 64 * 56 * 56 * 2 + 64 * 64 * 9 * 2 + 32 * 64 * 56 * 56 * 4,
        "strided": 32 * 256 * 28 * 28 * 2 + 256 * 128 * 9 * 2 + 32 * 128 * 56 * 56 * 4,
        "pointwise": 64 * 1024 * 14 * 14 * 2 + 1024 * 256 * 2 + 64 * 256 * 14 * 14 * 4,
        "stem": 16 * 64 * 112 * 112 * 4 + 64 * 3 * 49 * 4 + 16 * 3 * 224 * 224 * 4,
    }
    for key, nbytes in want.items():
        assert bench.algorithmic_bytes(workloads.BY_KEY[key]) == nbytes, key
    assert bench.algorithmic_bytes(workloads.RESNET) == 38_608_896


def test_useful_flops_closed_forms():
    # 2 * N * Co * OH * OW * Ci * kH * kW: every product of the definition once.
    assert bench.useful_flops(workloads.RESNET) == 2 * 32 * 64 * 56 * 56 * 64 * 9
    assert bench.useful_flops(workloads.STRIDED) == 2 * 32 * 256 * 28 * 28 * 128 * 9
    assert bench.useful_flops(workloads.POINTWISE) == 2 * 64 * 1024 * 14 * 14 * 256
    assert bench.useful_flops(workloads.STEM) == 2 * 16 * 64 * 112 * 112 * 3 * 49


def test_recorded_traffic_needs_the_same_kernel_source(monkeypatch, tmp_path):
    with open(bench.ROOT + "/profiles/dgrad_tc_resnet.traffic.json") as f:
        rec = json.load(f)
    assert rec["dram_bytes_per_launch"] == rec["dram_read_bytes"] + rec["dram_write_bytes"]
    monkeypatch.setattr(bench, "kernel_fingerprint", lambda: rec["kernel_fingerprint"])
    assert bench.recorded_traffic("resnet") == rec["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_fingerprint", lambda: "0" * 16)
    assert bench.recorded_traffic("resnet") is None
    assert bench.recorded_traffic("no-such-workload") is None

