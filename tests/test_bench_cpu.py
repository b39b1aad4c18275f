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



_NCU_HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
               '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
               '"Metric Value"')


def _ncu_row(i, name, metric, unit, value):
    return (f'"{i}","77","python3","127.0.0.1","{name}","1","13","(512, 1, 1)","(152, 1, 1)",'
            f'"0","10.3","Command line profiler metrics","{metric}","{unit}","{value}"')


def test_traffic_record_from_an_ncu_csv():
    k = "void dgrad::(anonymous namespace)::dgrad_tc_kernel<2, 1>(dgrad::TcParams)"
    rows = ["==PROF== Connected to process 77", _NCU_HEADER]
    # Launch 0 (cold: grad_in still in L2 at its end), then two steady launches.
    per = [(13_000_000, 2_304, 25_400), (13_100_000, 25_600_000, 17_900), (13_200_000, 25_800_000, 18_100)]
    for i, (rd, wr, ns) in enumerate(per):
        rows.append(_ncu_row(i, k, "dram__bytes_read.sum", "byte", f"{rd:,}"))
        rows.append(_ncu_row(i, k, "dram__bytes_write.sum", "byte", str(wr)))
        rows.append(_ncu_row(i, k, "gpu__time_duration.sum", "ns", str(ns)))
    rows.append(_ncu_row(9, "void other_kernel()", "dram__bytes_read.sum", "byte", "5"))
    launches = bench.traffic_from_ncu_csv("\n".join(rows))
    assert [x[0] for x in launches] == [0, 1, 2]
    assert launches[1][2:4] == (13_100_000, 25_600_000)
    assert launches[2][4] == pytest.approx(18.1e-6)
    rec = bench.traffic_record(launches, workloads.RESNET, "resnet", "cmd")
    # averaged over the launches after the first
    assert rec["dram_read_bytes"] == 13_150_000
    assert rec["dram_write_bytes"] == 25_700_000
    assert rec["dram_bytes_per_launch"] == 38_850_000
    assert rec["traffic_over_algorithmic"] == pytest.approx(38_850_000 / 38_608_896)
    assert rec["kernel"].startswith("dgrad::")
    # scaled units
    m = bench.traffic_from_ncu_csv("\n".join([
        _NCU_HEADER, _ncu_row(3, k, "dram__bytes_read.sum", "Mbyte", "1.5"),
        _ncu_row(3, k, "dram__bytes_write.sum", "Kbyte", "2")]))
    assert m[0][2:4] == (1_500_000, 2_000)


def test_shard_bounds_cover_the_batch_once():
    for n in (1, 7, 32, 64, 100):
        for world in (1, 2, 3, 4, 8):
            spans = [bench.shard_bounds(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_probes_compile_for_sm103a():
    # The device-rate probes bench.py --probe runs (cross-compiled here, no GPU).
    import shutil
    import subprocess
    import tempfile
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    for name, src in bench.PROBES.items():
        path = bench.ROOT + "/conv2d_backward_implicit_gb300/probes/" + src
        with tempfile.TemporaryDirectory() as d:
            r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                                path, "-o", d + "/" + name], capture_output=True, text=True)
            assert r.returncode == 0, r.stderr


def test_rmsnorm_flops_and_bytes():
    import bench
    f, b = bench.rmsnorm_flops_bytes(8192, 4096, 4096)
    assert f == 2.0 * 8192 * 4096 * 4096
    # X and W_proj bf16, W_norm bf16, C float32
    assert b == 8192 * 4096 * 2 + 4096 * 2 + 4096 * 4096 * 2 + 8192 * 4096 * 4
    assert bench.RMS_SHAPE["dtype"] == "bf16" and bench.RMS_SHAPE["n"] % 64 == 0 and bench.RMS_SHAPE["k"] % 8 == 0


def test_mha_useful_flops_counts_the_kept_pairs():
    import bench
    # causal 4 positions: 1 + 2 + 3 + 4 = 10 (query, key) pairs per head
    assert bench.mha_useful_flops(4, 0, 2, 8, 0) == 4 * 8 * 2 * 10
    # full attention 3 queries x 5 keys
    assert bench.mha_useful_flops(3, 5, 1, 4, 0) == 4 * 4 * 15
    # causal with window 2: 1 + 2 + 2 + 2
    assert bench.mha_useful_flops(4, 0, 1, 1, 2) == 4 * 7
    # brute force on a windowed full-attention case
    q, kv, w = 7, 5, 3
    pairs = sum(1 for pos in range(q) for t in range(kv) if t > pos - w)
    assert bench.mha_useful_flops(q, kv, 1, 1, w) == 4 * pairs
