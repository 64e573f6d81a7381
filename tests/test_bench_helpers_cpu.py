"""Host-side helpers of bench.py: the algorithmic quantizer bytes behind the
roofline fractions, the GEMM flop count, and the rule that a committed DRAM
traffic figure is reported only for the source it was captured on."""
import json
import os

import pytest

import bench


def test_quant_bytes_small_and_large_tensors():
    # a tensor within half the L2 is read once; a larger one twice (the
    # tensor amax is needed before any code is written)
    small = 1024 * 1024
    assert 2 * small <= 0.5 * bench.L2_BYTES
    assert bench.quant_bytes("quantize_1x16", 1024, 1024) == pytest.approx(small * (2 + 0.5 + 1 / 16))
    big_r, big_c = 8192, 11008
    n = big_r * big_c
    assert bench.quant_bytes("quantize_1x16", big_r, big_c) == pytest.approx(n * (4 + 0.5 + 1 / 16))
    # the dual and 2-D launches write two coded copies
    assert bench.quant_bytes("quantize_dual", big_r, big_c) == pytest.approx(n * (4 + 2 * (0.5 + 1 / 16)))
    assert bench.quant_bytes("quantize_2d_t", big_r, big_c) == pytest.approx(n * (4 + 2 * (0.5 + 1 / 16)))


def test_gemm_flops_of_the_step():
    assert bench.GEMM_FLOPS == 2 * 8192 * 11008 * 4096
    assert bench.N_GEMMS == 6


def test_traffic_reported_only_for_its_source():
    path = os.path.join(bench.ROOT, "profiles", "traffic.json")
    rec = json.load(open(path))["nvf4_gemm_pair_kernel"]
    assert bench.traffic_for("nvf4_gemm_pair_kernel", rec["source_hash"]) == pytest.approx(rec["dram_bytes_per_launch"])
    assert bench.traffic_for("nvf4_gemm_pair_kernel", "0" * 16) is None
    assert bench.traffic_for("no_such_kernel", rec["source_hash"]) is None
    # the hash covers every file the kernel is built from
    h = bench.source_hash(bench.GEMM_SOURCES)
    assert len(h) == 16 and all(os.path.exists(os.path.join(bench.ROOT, f)) for f in bench.GEMM_SOURCES)


def test_source_hash_follows_code_not_comments(tmp_path, monkeypatch):
    # the committed counters stay valid across comment edits and are dropped
    # by any change of code
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = tmp_path / "k.cu"
    f.write_text("int a = 1;  // one\n\n// note\nint b = 2;\n")
    h0 = bench.source_hash(["k.cu"])
    f.write_text("// header\nint a = 1;  // a different comment\nint b = 2;\n\n")
    assert bench.source_hash(["k.cu"]) == h0
    f.write_text("int a = 1;\nint b = 3;\n")
    assert bench.source_hash(["k.cu"]) != h0

