"""Host-side arithmetic of bench.py: the roofline fields, the launch count per
call and the hash-keyed traffic records (no GPU)."""
import json
import os

import pytest

import bench

PEAKS = {"bf16_tflops": 1887.4, "source": "MEASURED_PEAKS.json", "sm_max_mhz": 2070.0,
         "tf32_tflops": 1185.8, "tf32_n128_tflops": 844.0, "bf16_n128_tflops": 1707.0}
FLOPS = 51_547_996_160.0  # the serving chunk: 4 * 64 * 32 * pairs


def test_split_tf32_roofline_fields():
    r = bench.roofline("attn_prefill", "tcgen05-split-tf32", FLOPS, 0.2062, PEAKS, "serve")
    achieved = FLOPS / 0.2062e-3 / 1e12
    assert r["bound"] == "tensor" and r["peak_dtype"] == "tf32" and r["tensor_passes"] == 3
    assert r["peak"] == pytest.approx(1185.8)
    assert r["frac"] == pytest.approx(achieved / 1185.8, abs=1e-4)
    assert r["frac_of_split_roof"] == pytest.approx(3 * achieved / 1185.8, abs=1e-4)
    assert r["tensor_work_frac_of_n128_loop"] == pytest.approx(3 * achieved / 844.0, abs=1e-4)
    # the older denominator, the measured bf16 burst scaled by the nominal tf32/bf16 ratio
    assert r["peak_nominal_ratio"] == pytest.approx(1887.4 * 1.1 / 2.25, abs=1e-3)


def test_bf16_roofline_fields():
    for kernel, passes in (("tcgen05-bf16x3", 3), ("tcgen05-bf16kv", 2)):
        r = bench.roofline("attn_prefill_bf16x3", kernel, FLOPS, 0.156, PEAKS, "serve")
        achieved = FLOPS / 0.156e-3 / 1e12
        assert r["tensor_passes"] == passes and r["peak"] == pytest.approx(1887.4)
        assert r["frac_of_split_roof"] == pytest.approx(passes * achieved / 1887.4, abs=1e-4)
        assert r["tensor_work_frac_of_n128_loop"] == pytest.approx(passes * achieved / 1707.0, abs=1e-4)


def test_roofline_without_a_live_tensor_peak():
    peaks = {k: v for k, v in PEAKS.items() if k not in ("tf32_tflops", "tf32_n128_tflops", "bf16_n128_tflops")}
    r = bench.roofline("attn_prefill", "tcgen05-split-tf32", FLOPS, 0.2062, peaks, "serve")
    assert r["peak"] == pytest.approx(1887.4 * 1.1 / 2.25, abs=1e-3)  # the nominal-ratio fallback
    assert "tensor_work_frac_of_n128_loop" not in r


def test_ffma_roofline_is_the_fp32_pipe():
    r = bench.roofline("attn_prefill_ffma", "ffma", FLOPS, 1.302, PEAKS, "serve")
    assert r["bound"] == "alu"
    assert r["peak"] == pytest.approx(152 * 128 * 2 * 2070e6 / 1e12, abs=1e-3)


@pytest.mark.parametrize("path,C,P,launches", [
    ("attn_prefill", 2048, 2048, 2),      # three full rounds, then 56 units split over pairs
    ("attn_prefill", 2048, 30720, 2),
    ("attn_prefill", 256, 32768, 1),      # 64 units: all split in one pair grid
    ("attn_prefill", 608, 0, 1),          # exactly one round
    ("attn_prefill", 640, 0, 1),          # the shortest unit sees fewer than 1024 keys
    ("attn_prefill_bf16kv", 2048, 2048, 2),  # the bf16 paths take the same last-round rule
    ("attn_prefill_bf16kv", 2048, 30720, 2),
    ("attn_decode_paged", 16, 16384, 1),
    ("attn_prefill", 928, 8192, 2),       # a last round of 80 units over threes in two waves
    ("attn_prefill", 928, 4096, 1),       # the same units too short for it: whole units
])
def test_launches_per_call(path, C, P, launches):
    assert bench.launches_per_call(path, C, P) == launches


def test_traffic_record_goes_stale_with_its_source(tmp_path, monkeypatch):
    csrc = tmp_path / "chunked_prefill_gqa_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "tc.cu").write_text("// kernel source as profiled\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    record = {"attn_prefill:serve": {"dram_bytes_per_launch": 33690624,
                                     "source_sha256_16": bench.kernel_source_hash("attn_prefill")}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(record))
    assert bench.profiled_traffic("attn_prefill", "serve") == 33690624
    assert bench.profiled_traffic("attn_prefill", "long") is None  # no record for that workload
    (csrc / "tc.cu").write_text("// kernel source changed since the capture\n")
    assert bench.profiled_traffic("attn_prefill", "serve") is None


def test_chunk_workload_metric_and_row_sample():
    import argparse
    a = argparse.Namespace(workload="chunk", chunk=32, prefix=32768)
    assert bench.metric_for(a).startswith("attention TFLOP/s at C=32,P=32768 ")
    assert bench.metric_for(argparse.Namespace(workload="serve", chunk=0, prefix=0)) == bench.METRIC
    assert bench.sample_rows_for_cpu(32, 64) == [31]  # fewer rows than the stride: the last row
    assert bench.sample_rows_for_cpu(130, 64) == [63, 127, 129]
