"""Shared helpers for the GPU tests: seeded workloads, the oracle on a subset
of rows, and the acceptance tolerances.

Tolerances (logits): bf16 models max |dlogit| <= 3e-2 and mean |dlogit| <= 5e-3;
fp32 model max |dlogit| <= 1e-4.
"""
import numpy as np
import torch

import nc_inputs
from oracle.gpt_oracle import OracleModel

TOL = {"bf16": (3e-2, 5e-3), "f32": (1e-4, 1e-4)}


def small_bf16_shape(n_layer=2, vocab=4096):
    """d12 widths (d 768, 6 heads of 128, MLP 3072) with fewer layers and a smaller vocabulary."""
    return nc_inputs.D12.with_(name="d12_small", n_layer=n_layer, vocab=vocab)


def check_close(got, want, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU values"
    err = np.abs(got - want)
    mx, mean = float(err.max()), float(err.mean())
    tmax, tmean = TOL[dtype]
    assert mx <= tmax and mean <= tmean, f"{what}: max {mx:.3e} (tol {tmax}), mean {mean:.3e} (tol {tmean})"
    return mx, mean


def tokens_for(w):
    """Prompt [B, T] and decode tokens [steps, B] of a workload."""
    V = w.shape.vocab
    prompt = nc_inputs.gen_tokens(V, (w.batch, w.prompt_len), w.prompt_seed)
    nxt = (nc_inputs.gen_tokens(V, (w.decode_steps, w.batch), w.decode_seed)
           if w.decode_steps else np.zeros((0, w.batch), np.int32))
    return prompt, nxt


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def oracle_for(flat, shape):
    return OracleModel(flat, shape)
