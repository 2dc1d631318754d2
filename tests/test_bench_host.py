"""bench.py's algorithmic work counts (the numerators of every roofline
fraction it reports) against totals derived independently from the model
configurations: the parameter counts of the blocks and of the unembedding,
and the causal attention pair count.

Expected values (hand-derived from the configs, 2 FLOPs per MAC, one KV head):
  parameters per block = d (n_h + 2) 128 + n_h 128 d + 2 d F, unembedding V d;
  prefill FLOPs = 2 M (L block + V d) + 4 n_h 128 T (T + 1) / 2 B L;
  decode bytes per step = bf16 weights once + K/V read at the step's context +
  one K/V row written + embedding rows + fp32 logits.
"""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import nc_inputs  # noqa: E402

# parameters of the blocks (all layers) and of one of E / Wu, one KV head
BLOCK_PARAMS = {"d12": 73_138_176, "d20": 334_233_600, "d24": 575_668_224}
UNEMBED_PARAMS = {"d12": 50_331_648, "d20": 83_886_080, "d24": 100_663_296}


@pytest.mark.parametrize("name,shape", [("d12", nc_inputs.D12), ("d20", nc_inputs.D20), ("d24", nc_inputs.D24)])
def test_parameter_counts_of_the_configs(name, shape):
    d, nh, F, V, L = shape.d_model, shape.n_head, shape.d_mlp, shape.vocab, shape.n_layer
    assert L * (d * (nh + 2) * 128 + nh * 128 * d + 2 * d * F) == BLOCK_PARAMS[name]
    assert V * d == UNEMBED_PARAMS[name]


@pytest.mark.parametrize("name,shape,B,T,tflop", [
    ("d12", nc_inputs.D12, 8, 2048, 4.665),
    ("d20", nc_inputs.D20, 16, 2048, 30.84),
    ("d24", nc_inputs.D24, 8, 2048, 24.64),
])
def test_prefill_flops_match_the_stated_totals(name, shape, B, T, tflop):
    f = bench.prefill_flops(shape, B, T)
    M = B * T
    attn = 4.0 * shape.n_head * 128 * (T * (T + 1) / 2) * B * shape.n_layer
    total = 2.0 * M * (BLOCK_PARAMS[name] + UNEMBED_PARAMS[name]) + attn
    assert sum(f.values()) == pytest.approx(total, rel=1e-12)
    assert sum(f.values()) / 1e12 == pytest.approx(tflop, abs=0.006)
    # last-position logits only: the unembedding shrinks from M rows to B rows
    g = bench.prefill_flops(shape, B, T, last_only=True)
    assert f["lm_head"] - g["lm_head"] == pytest.approx(2.0 * (M - B) * UNEMBED_PARAMS[name])


@pytest.mark.parametrize("name,shape,B,ctx0,steps,mbytes", [
    ("d12", nc_inputs.D12, 32, 512, 256, 381.5),
    ("d20", nc_inputs.D20, 64, 1024, 128, 1567.0),
    ("d24", nc_inputs.D24, 128, 2048, 128, 4711.0),
])
def test_decode_bytes_match_the_stated_totals(name, shape, B, ctx0, steps, mbytes):
    ctxs = [ctx0 + t + 1 for t in range(steps)]
    got = np.mean([bench.decode_bytes(shape, B, c) for c in ctxs])
    L, d, V = shape.n_layer, shape.d_model, shape.vocab
    kv_row = 2 * 128 * 2                                    # K and V, 128 dims, bf16
    want = np.mean([2.0 * (BLOCK_PARAMS[name] + UNEMBED_PARAMS[name])
                    + L * B * c * kv_row + L * B * kv_row + B * d * 2 + B * V * 4 for c in ctxs])
    assert got == pytest.approx(want, rel=1e-12)
    assert got / 1e6 == pytest.approx(mbytes, abs=0.6)


def test_decode_bytes_with_fp8_weights():
    """FP8 workload: every projection weight (blocks and unembedding) is one
    byte; the K/V cache, embedding rows and logits are unchanged."""
    s8 = nc_inputs.D24.with_(dtype="fp8")
    B, ctx = 128, 2100
    L, d, V = s8.n_layer, s8.d_model, s8.vocab
    kv_row = 2 * 128 * 2
    want = (1.0 * (BLOCK_PARAMS["d24"] + UNEMBED_PARAMS["d24"]) + L * B * ctx * kv_row + L * B * kv_row
            + B * d * 2 + B * V * 4)
    assert bench.decode_bytes(s8, B, ctx) == pytest.approx(want, rel=1e-12)
    assert bench.decode_bytes(nc_inputs.D24, B, ctx) - bench.decode_bytes(s8, B, ctx) == pytest.approx(
        BLOCK_PARAMS["d24"] + UNEMBED_PARAMS["d24"], rel=1e-12)
    # resident weights: bf16 embedding table plus one byte per projection weight
    assert bench.weight_bytes(s8) == 2 * V * d + BLOCK_PARAMS["d24"] + UNEMBED_PARAMS["d24"]


def test_work_counts_with_grouped_query_heads():
    """n_kv K/V heads: the QKV projection grows by 2 (n_kv - 1) heads, the
    K/V cache traffic by a factor n_kv; the attention FLOPs (one score and
    one output product per query head) do not change."""
    s1 = nc_inputs.D12
    s3 = nc_inputs.D12.with_(n_kv_head=3)
    B, T, ctx = 4, 512, 700
    d, L = s1.d_model, s1.n_layer
    f1, f3 = bench.prefill_flops(s1, B, T), bench.prefill_flops(s3, B, T)
    assert f3["qkv"] - f1["qkv"] == pytest.approx(2.0 * B * T * d * (2 * 2 * 128) * L)
    assert f3["attn"] == f1["attn"]
    b1, b3 = bench.decode_bytes_by_class(s1, B, ctx), bench.decode_bytes_by_class(s3, B, ctx)
    assert b3["attn"] == pytest.approx(3 * b1["attn"])
    assert b3["qkv"] - b1["qkv"] == pytest.approx(2.0 * L * (2 * 2 * 128) * d + L * B * 2 * 2 * 128 * 2.0)

