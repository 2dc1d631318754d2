"""GPU parity at the d20 and d24 workloads, in the launch configuration the
benchmark uses (full batch, full length), against the fp64 oracle on sampled
rows: rows are independent, so the oracle recomputes a few of them exactly.

Prefill: rows 0 and B-1 at every position.  Decode: the full batch decodes
every step through the captured CUDA graph (one fixed logits buffer), and
rows 0, B/2 and B-1 are checked at every step.

Tolerances (logits): max |dlogit| <= 3e-2 and mean |dlogit| <= 5e-3 (bf16).
"""
import numpy as np
import pytest
import torch

import dense_gpt_transformer_fwd_b300 as ncp
import nc_inputs
from nc_testutil import check_close, oracle_for, to_dev, tokens_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gpt_transformer_fwd_b300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("name", ["d20_prefill", "d24_prefill"])
def test_prefill_full_size_sampled_rows(name):
    w = nc_inputs.WORKLOADS[name]
    flat = nc_inputs.gen_weights(w.shape, w.weight_seed)
    prompt, _ = tokens_for(w)
    rows = [0, w.batch - 1]
    m = ncp.Model(w.shape, flat, max_batch=w.batch, max_seq=w.max_seq)
    got = m.prefill(to_dev(prompt))
    m.sync()
    sample = got[rows].cpu().numpy()
    finite = bool(torch.isfinite(got).all())
    m.close()
    del got
    torch.cuda.empty_cache()
    assert finite
    want = oracle_for(flat, w.shape).prefill(prompt[rows])
    check_close(sample, want, "bf16", f"{name} rows {rows}")


@pytest.mark.parametrize("name", ["d20_decode", "d24_decode"])
def test_decode_full_size_sampled_rows(name):
    w = nc_inputs.WORKLOADS[name]
    flat = nc_inputs.gen_weights(w.shape, w.weight_seed)
    prompt, nxt = tokens_for(w)
    rows = [0, w.batch // 2, w.batch - 1]
    m = ncp.Model(w.shape, flat, max_batch=w.batch, max_seq=w.max_seq)
    m.prefill(to_dev(prompt), last_only=True)
    out = torch.empty((w.batch, w.shape.vocab), device="cuda")
    nxt_d = to_dev(nxt)
    got = []
    for t in range(w.decode_steps):
        m.decode_step(nxt_d[t], out=out)
        got.append(out[rows].cpu().numpy())
    m.sync()
    assert m.kv_length() == (w.max_seq, w.batch)
    m.close()
    torch.cuda.empty_cache()
    o = oracle_for(flat, w.shape)
    o.prefill(prompt[rows], logit_positions=[w.prompt_len - 1])
    for t in range(w.decode_steps):
        check_close(got[t], o.decode(nxt[t][rows]), "bf16", f"{name} step {t}")
