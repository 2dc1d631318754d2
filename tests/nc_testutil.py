"""Shared helpers for the GPU tests: seeded workloads, the oracle on a subset
of rows, and the acceptance tolerances.

Tolerances (logits): bf16 models max |dlogit| <= 3e-2 and mean |dlogit| <= 5e-3;
fp32 model max |dlogit| <= 1e-4.
"""
import re

import numpy as np
import torch

import nc_inputs
from oracle.gpt_oracle import OracleModel

TOL = {"bf16": (3e-2, 5e-3), "f32": (1e-4, 1e-4)}


def small_bf16_shape(n_layer=2, vocab=4096):
    """d12 widths (d 768, 6 heads of 128, MLP 3072) with fewer layers and a smaller vocabulary."""
    return nc_inputs.D12.with_(name="d12_small", n_layer=n_layer, vocab=vocab)


# worst margins per check group, printed at the end of the session (conftest)
MARGINS = {}


def _record(group, mx, mean, tmax, tmean):
    old = MARGINS.get(group)
    if old is None:
        MARGINS[group] = (mx, mean, tmax, tmean, 1)
    else:
        MARGINS[group] = (max(old[0], mx), max(old[1], mean), tmax, tmean, old[4] + 1)


def check_close(got, want, dtype, what="", group=None, tol=None):
    """max and mean |got - want| within the tolerance of `dtype` (or `tol`);
    the margins are recorded under `group` (default: `what` without a
    trailing step number) for the end-of-session summary."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU values"
    err = np.abs(got - want)
    mx, mean = float(err.max()), float(err.mean())
    tmax, tmean = tol if tol is not None else TOL[dtype]
    if group is None:
        group = re.sub(r"\s*\d+$", "", what) or what      # "d12 decode step 5" -> "d12 decode step"
        if tol is None:
            group += f" [{dtype}]"
    _record(group, mx, mean, tmax, tmean)
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
