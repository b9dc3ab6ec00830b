"""bench.py's host-side pieces on CPU: the per-stage byte model agrees with the algorithmic
bytes per token of the scope table, the CPU baseline times the oracle in child processes on one
core and on all cores, and the replica arithmetic."""
import os

import pytest

from engram_synth import get_workload
from engram_synth.case import make_case
from oracle import engram_oracle as O

import bench

PEAKS = {"hbm_gbs": 6780.4, "bf16_tflops": 1923.3, "bf16_tflops_sustained": 1712.0}


@pytest.mark.parametrize("name,gather_per_token,gate_per_token", [
    ("decode_fp8_t256", 18720, 172032), ("prefill_fp8_t32768", 18720, 172032),
    ("large_fp8_t16384", 18720, 301056), ("q2k_t8192", 14400, 172032), ("tiny_bf16", 1024 + 32 + 1024, 10752)])
def test_stage_bytes_per_token(name, gather_per_token, gate_per_token):
    w = get_workload(name)
    T, N, K, H, hc = w.tokens, w.N, w.K, w.hidden, w.hc
    g = bench.stage_model(w, "gather0", PEAKS)
    assert g["bytes"] == gather_per_token * T
    ga = bench.stage_model(w, "gate0", PEAKS)
    assert ga["bytes"] - 4 * hc * H == gate_per_token * T          # + the q/k weights once per launch
    assert ga["extra_bytes"] == 2 * N * T                          # fp32 kv read instead of bf16
    p = bench.stage_model(w, "project0", PEAKS)
    assert p["bytes"] == 2 * N * K + 2 * K * T + 2 * N * T and p["flops"] == 2 * T * N * K
    assert p["extra_bytes"] == 2 * N * T


def test_projection_bound_follows_the_ridge():
    assert bench.stage_model(get_workload("decode_fp8_t256"), "project0", PEAKS)["bound"] == "hbm"
    assert bench.stage_model(get_workload("large_fp8_t16384"), "project0", PEAKS)["bound"] == "tensor"
    assert bench.stage_model(get_workload("large_fp8_t64"), "project0", PEAKS)["bound"] == "hbm"


def test_headline_workload_is_the_largest_configuration():
    assert bench.DEFAULT_WORKLOAD == "large_fp8_t16384"


def test_roofline_entry_carries_both_denominators():
    w = get_workload("large_fp8_t16384")
    m = bench.stage_model(w, "project0", PEAKS)
    r = bench.roofline_entry("project0", m, 1700.0, PEAKS["bf16_tflops"], "TFLOP/s", PEAKS, "measured", False, None)
    assert r["frac"] == round(1700.0 / 1923.3, 4) and r["frac_sustained"] == round(1700.0 / 1712.0, 4)
    m = bench.stage_model(w, "gate0", PEAKS)
    r = bench.roofline_entry("gate0", m, 6000.0, PEAKS["hbm_gbs"], "GB/s", PEAKS, "measured", False, None)
    assert r["frac_nominal"] == round(6000.0 / bench.NOMINAL_HBM_GBS, 4)


def test_replica_throughput():
    assert bench.replica_throughput(4, 1000, 2.0) == 4 * 1000 / 0.002
    assert bench.max_over_ranks(3.5, "cpu") == 3.5


def test_cpu_baseline_times_the_oracle_on_one_and_all_cores():
    w = get_workload("tiny_bf16")
    _, _, rows = O.layout(w.vocab_size, w.layers, w.max_ngram, w.n_heads)
    case = make_case(w, [int(r) for r in rows], "cpu")
    out = bench.cpu_baseline(w, case, 8, seconds=0.2)
    assert out["kind"] == "oracle" and out["unit"] == "tokens/s per layer"
    assert out["one_core"]["cores"] == 1 and out["all_cores"]["cores"] == (os.cpu_count() or 1)
    assert out["one_core"]["value"] > 0 and out["value"] == out["all_cores"]["value"]


def test_mxfp8_peak_is_the_measured_one():
    assert bench.tensor_peak(PEAKS, True) == bench.MXFP8_PEAK_TFLOPS["burst"]
    assert bench.tensor_peak(PEAKS, False) == PEAKS["bf16_tflops"]
    assert bench.tensor_peak(PEAKS, False, "sustained") == PEAKS["bf16_tflops_sustained"]
