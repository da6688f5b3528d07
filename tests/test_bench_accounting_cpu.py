"""The work bench.py divides by: algorithmic bytes and flops per step, pinned to independent counts.

The projection weights a step streams are every layer's four matrices plus the tied head.
Adding back what the bench leaves out (biases, norm gains and biases, learned positions) must
give each model's published total parameter count exactly, so a wrong shape, a dropped matrix
or a miscounted head dimension fails here.
"""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
import workloads as wl  # noqa: E402


def _gpt2_extra(s):   # per layer: ln1 (2d), qkv bias, o bias, ln2 (2d), up bias (F), down bias; lnf; positions
    d = s.d_model
    per_layer = 2 * d + s.qkv_dim + d + 2 * d + s.d_ff + d
    return s.n_layers * per_layer + 2 * d + s.n_ctx * d


def _llama_extra(s):  # per layer: two RMSNorm gains; final norm gain
    return s.n_layers * 2 * s.d_model + s.d_model


@pytest.mark.parametrize("shape,extra,total", [
    (wl.GPT2_124M_F32, _gpt2_extra, 124_439_808),
    (wl.SMOLLM2_360M, _llama_extra, 361_821_120),
    (wl.GPT2_XL_BF16, _gpt2_extra, 1_557_611_200),
], ids=["gpt2-124m", "smollm2-360m", "gpt2-xl"])
def test_streamed_weights_plus_the_rest_are_the_published_parameter_count(shape, extra, total):
    streamed = bench.weight_bytes(shape) // shape.elt_bytes
    assert streamed + extra(shape) == total


def test_gpt2_124m_fp32_step_bytes_by_hand():
    s, B = wl.GPT2_124M_F32, 32
    weights = (12 * (2304 * 768 + 768 * 768 + 3072 * 768 + 768 * 3072) + 50257 * 768) * 4
    assert bench.weight_bytes(s) == weights == 494_128_128
    # activations per layer: qkv x in + q,k,v out; o x in + residual read and write; up; down;
    # and the head's normalised input
    acts = 12 * B * ((768 + 2304) * 4 + (768 + 2 * 768) * 4 + (768 + 3072) * 4 + (3072 + 2 * 768) * 4) + B * 768 * 4
    assert bench.gemv_bytes(s, B) == weights + acts
    ctx = np.array([129, 200, 256], dtype=np.int64)
    kv = int(ctx.sum()) * 12 * 64 * 4 * 2 * 12
    assert bench.attn_bytes(s, ctx) == kv + 3 * 12 * 64 * 8 * 12
    assert bench.step_bytes(s, ctx) == bench.gemv_bytes(s, 3) + bench.attn_bytes(s, ctx)


def test_prefill_flops_by_hand():
    s = wl.GPT2_124M_BF16
    lengths = np.full(16, 1024)
    proj = 2.0 * 16 * 1024 * 12 * (2304 * 768 + 768 * 768 + 3072 * 768 + 768 * 3072) + 2.0 * 16 * 50257 * 768
    assert bench.prefill_gemm_flops(s, lengths) == pytest.approx(proj, rel=1e-15)
    pairs = 16 * 1024 * 1025 // 2
    assert bench.prefill_attn_flops(s, lengths) == pytest.approx(4.0 * pairs * 64 * 12 * 12, rel=1e-15)


def test_traffic_table_matches_only_its_own_kernel_family():
    for name, (family, value) in bench.TRAFFIC.items():
        assert name in wl.WORKLOADS
        assert bench.traffic_for(name, family) == value > 0
        assert bench.traffic_for(name, family + " (other)") is None


def test_family_roofline_never_charges_more_than_the_step():
    import bench
    # long kernels: the event-timed duration fits in the step and is used as measured
    fams = {"attn_decode": [48, 10.0], "proj": [196, 4.0]}
    r = bench.family_roofline(fams, "attn_decode", 1, 15.0, 48 * 1e9, "GB/s", 6000.0, "x", "attn", None)
    assert r["duration_method"].startswith("CUDA events")
    assert abs(r["avg_launch_us"] - 10.0e3 / 48) < 1e-9
    assert abs(r["achieved"] - 1e9 / (10.0e-3 / 48) / 1e9) < 1e-6
    # short kernels whose event intervals add launch latency: the family's event time per step
    # (0.7 ms) exceeds the timed step (0.55 ms), so it is charged its share of the step
    fams = {"proj": [49, 0.70], "norm": [25, 0.20], "attn_decode": [12, 0.10]}
    r = bench.family_roofline(fams, "proj", 1, 0.55, 49 * 10e6, "GB/s", 6000.0, "x", "proj", None)
    assert r["duration_method"].startswith("share")
    assert abs(r["family_ms_per_step"] - 0.55 * 0.7) < 1e-12
    assert r["family_ms_per_step"] <= 0.55
    assert abs(r["frac"] - r["achieved"] / 6000.0) < 1e-12
