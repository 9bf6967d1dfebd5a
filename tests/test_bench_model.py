"""The benchmark's algorithmic work model (the numerator of every roofline fraction) against
closed forms: FLOPs are twice the layer's active parameters per token (2*M*N*K per GEMM);
bytes are the weights read once plus the input and output rows.  CPU only."""
import pytest

import bench
from workloads import WORKLOADS

FULL = WORKLOADS["full_prefill_bt8192"].shape

# active parameters per token of the full-width layer: router 896 x 7168, W_down and W_up
# 7168 x 3584 each, 16 experts of 3 x 3584 x 3072, 2 shared experts of 3 x 7168 x 3072
ACTIVE = 896 * 7168 + 2 * 7168 * 3584 + 16 * 3 * 3584 * 3072 + 2 * 3 * 7168 * 3072
# all weights of the layer in bf16, plus the RMSNorm gain
WEIGHT_BYTES = 2 * (896 * 7168 + 2 * 7168 * 3584 + 3584 + 896 * 3 * 3584 * 3072 + 2 * 3 * 7168 * 3072)


def test_flops_per_token_is_twice_the_active_parameters():
    assert 2 * ACTIVE == 1_436_811_264
    for bt in (1, 64, 8192, 16384):
        flops, _, stages = bench.algorithmic(FULL, bt, FULL.n_experts)
        assert flops == 2 * ACTIVE * bt
        assert sum(f for f, _ in stages.values()) == flops
    assert bench.algorithmic(FULL, 8192, 896)[0] == pytest.approx(11.77e12, rel=1e-3)
    assert bench.algorithmic(FULL, 64, 613)[0] == pytest.approx(91.96e9, rel=1e-3)


def test_layer_bytes_are_the_weights_plus_rows_in_and_out():
    _, b, _ = bench.algorithmic(FULL, 8192, 896)
    assert b == WEIGHT_BYTES + 2 * 8192 * 7168 * 2
    assert WEIGHT_BYTES == pytest.approx(59.57e9, rel=1e-3)
    assert b == pytest.approx(59.80e9, rel=1e-3)
    # untouched experts are not read: each one missing saves its 3 x 3584 x 3072 bf16 weights
    _, b_dec, _ = bench.algorithmic(FULL, 64, 820)
    assert b - b_dec == (896 - 820) * 3 * 3584 * 3072 * 2 + 2 * (8192 - 64) * 7168 * 2


def test_dominant_stage_units():
    """The per-launch units quoted for the expert GEMMs at 8192 tokens: the weights of all 896
    experts (token rows and activations are intermediates of the layer, not counted)."""
    _, _, st = bench.algorithmic(FULL, 8192, 896)
    f, b = st["expert_gate_up_gemm"]
    assert f == 2 * 8192 * 16 * 2 * 3072 * 3584
    assert b == 896 * 2 * 3072 * 3584 * 2
    assert b == pytest.approx(39.46e9, rel=1e-3)
    assert st["expert_down_gemm"][1] == pytest.approx(19.73e9, rel=1e-3)
    # the two expert stages together carry the layer's expert weight bytes
    _, layer, _ = bench.algorithmic(FULL, 8192, 896)
    assert b + st["expert_down_gemm"][1] == 896 * 3 * 3584 * 3072 * 2 < layer


def test_fp8_experts_byte_model():
    """e4m3 experts: one byte per expert weight plus a 4-byte scale per output row; the rest of
    the layer stays bf16; FLOPs are unchanged."""
    f16, b16, _ = bench.algorithmic(FULL, 8192, 896)
    f8, b8, st8 = bench.algorithmic(FULL, 8192, 896, fp8_experts=True)
    assert f8 == f16
    expert_params = 896 * 3 * 3584 * 3072
    scales = 896 * (2 * 3072 + 3584) * 4
    assert b16 - b8 == expert_params - scales
    g = st8["expert_gate_up_gemm"][1]
    assert g == 896 * 2 * 3072 * (3584 + 4)


def test_mxfp4_experts_byte_model():
    """MXFP4 experts: half a byte per expert weight plus one scale byte per 32 weights (17/32 byte
    per weight, 29.6 G weights -> 15.7 GB); the rest of the layer stays bf16; FLOPs are unchanged."""
    f16, b16, _ = bench.algorithmic(FULL, 8192, 896)
    f4, b4, st4 = bench.algorithmic(FULL, 8192, 896, mxfp4_experts=True)
    assert f4 == f16
    expert_params = 896 * 3 * 3584 * 3072
    assert b16 - b4 == pytest.approx(expert_params * (2 - 17 / 32), rel=1e-12)
    assert st4["expert_gate_up_gemm"][1] == pytest.approx(896 * 2 * 3072 * 3584 * 17 / 32, rel=1e-12)
    assert st4["expert_gate_up_gemm"][1] + st4["expert_down_gemm"][1] == pytest.approx(15.73e9, rel=1e-3)


def test_layer_fraction_takes_the_binding_roof():
    """The layer line's `bound` is the roof with the larger ideal time and `frac` its fraction:
    at 8192 tokens the 59.8 GB of weights and rows bind (HBM), at 16384 the 23.5 TFLOP do."""
    pk = {"hbm": 6500.0, "tc": 1756.5}
    r = bench.layer_fractions(FULL, 8192, 896, 0.0154, pk)
    assert r["bound"] == "hbm" and r["frac"] == r["hbm_frac"]
    assert r["hbm_frac"] == pytest.approx(59.80e9 / 0.0154 / 6500e9, rel=1e-3)
    assert r["tc_frac"] == pytest.approx(11.77e12 / 0.0154 / 1756.5e12, rel=1e-3)
    r = bench.layer_fractions(FULL, 16384, 896, 0.030, pk)
    assert r["bound"] == "tensor" and r["frac"] == r["tc_frac"]


def test_traffic_record_applies_only_to_its_workload_and_format():
    """roofline.traffic comes from the committed ncu record only for the launch it was scaled to
    (workload and expert format) and only while the kernel source is the one it was taken from."""
    import json
    import os
    rec = json.load(open(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")))["expert_gate_up_gemm"]
    got = bench.kernel_traffic("expert_gate_up_gemm", rec["workload"], rec["experts"])
    assert got in (None, rec["dram_bytes_per_launch"])   # None once the kernel source has changed
    assert bench.kernel_traffic("expert_gate_up_gemm", "full_decode_bt64", rec["experts"]) is None
    assert bench.kernel_traffic("expert_gate_up_gemm", rec["workload"], "mxfp4") is None
    assert bench.kernel_traffic("router_gemm", rec["workload"], rec["experts"]) is None
