"""The later-architecture extras on the GPU (value embeddings, residual/x0
lambdas, smear, backout; apidog.com/th "how nanochat works" item 1), through
the C ABI, against the fp64 oracle on the same seeded inputs.  On synthetic
weights these are parity checks only: the pages' trained values are not
available.  Tolerances: bf16 max 3e-2 / mean 5e-3, fp32 1e-4.
"""
import numpy as np
import pytest
import torch

import dense_gpt_transformer_fwd_b300 as ncp
import nc_inputs
from nc_testutil import check_close, oracle_for, small_bf16_shape, to_dev

pytestmark = pytest.mark.gpu

ALL = dict(value_embeds=True, resid_lambdas=True, smear=True, backout=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gpt_transformer_fwd_b300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_every_extra_prefill_decode_chunk_clone(dtype):
    if dtype == "bf16":
        sh = small_bf16_shape(n_layer=3, vocab=2048).with_(n_kv_head=2, **ALL)
    else:
        sh = nc_inputs.TINY.with_(**ALL)
    flat = nc_inputs.gen_weights(sh, 210)
    B, T = 2, 150
    toks = nc_inputs.gen_tokens(sh.vocab, (B, T + 3 + 40 + 2), 211)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + 3 + 40 + 2)
    tag = f"extras {dtype}"
    check_close(m.prefill(to_dev(toks[:, :T])).cpu().numpy(), o.prefill(toks[:, :T]), dtype, f"{tag}: prefill")
    p = T
    for _ in range(3):
        check_close(m.decode_step(to_dev(toks[:, p])).cpu().numpy(), o.decode(toks[:, p]), dtype, f"{tag}: decode")
        p += 1
    check_close(m.prefill(to_dev(toks[:, p:p + 40])).cpu().numpy(), o.extend(toks[:, p:p + 40]), dtype,
                f"{tag}: chunk")
    p += 40
    m.kv_clone(1, 2)
    o.clone_row(1, 2)
    for _ in range(2):
        check_close(m.decode_step(to_dev(toks[:, p])).cpu().numpy(), o.decode(toks[:, p]), dtype,
                    f"{tag}: decode after a clone")
        p += 1
    m.sync()
    m.close()


@pytest.mark.parametrize("which", ["value_embeds", "resid_lambdas", "smear", "backout"])
def test_each_extra_alone(which):
    sh = small_bf16_shape(n_layer=2, vocab=2048).with_(**{which: True})
    flat = nc_inputs.gen_weights(sh, 212)
    B, T = 3, 70
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 213)
    nxt = nc_inputs.gen_tokens(sh.vocab, (2, B), 214)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + 2)
    check_close(m.prefill(to_dev(prompt)).cpu().numpy(), o.prefill(prompt), "bf16", f"extra {which}: prefill")
    for t in range(2):
        check_close(m.decode_step(to_dev(nxt[t])).cpu().numpy(), o.decode(nxt[t]), "bf16",
                    f"extra {which}: decode")
    m.sync()
    m.close()


def test_smear_with_rows_of_different_lengths():
    """Each row's smear reaches back to its own last token across calls."""
    sh = small_bf16_shape(n_layer=2, vocab=2048).with_(**ALL)
    flat = nc_inputs.gen_weights(sh, 215)
    B, T = 3, 60
    lens = [60, 17, 1]
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 216)
    nxt = nc_inputs.gen_tokens(sh.vocab, (2, B), 217)
    orc = [oracle_for(flat, sh) for _ in range(B)]
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + 2)
    got = m.prefill_rows(to_dev(prompt), lens, last_only=True).cpu().numpy()
    for b in range(B):
        want = orc[b].prefill(prompt[b:b + 1, :lens[b]], logit_positions=[lens[b] - 1])[0, 0]
        check_close(got[b], want, "bf16", "extras ragged rows: prefill")
    for t in range(2):
        got = m.decode_step(to_dev(nxt[t])).cpu().numpy()
        for b in range(B):
            check_close(got[b], orc[b].decode(nxt[t][b:b + 1])[0], "bf16", "extras ragged rows: decode")
    m.sync()
    m.close()


def test_extras_with_fp8_weights_groups_and_windows():
    """Every extra together with FP8 projection weights, three K/V heads and
    a window on alternate layers: prefill, decode steps (the generic decode
    path, since the extras keep the decode graph off) and a chunk, against
    the oracle on the same rounded weights."""
    sh = small_bf16_shape(n_layer=4, vocab=2048).with_(dtype="fp8", n_kv_head=3, window=100, window_pattern="SL",
                                                        **ALL)
    flat = nc_inputs.gen_weights(sh, 218)
    B, T = 2, 180
    toks = nc_inputs.gen_tokens(sh.vocab, (B, T + 3 + 30), 219)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + 3 + 30)
    check_close(m.prefill(to_dev(toks[:, :T])).cpu().numpy(), o.prefill(toks[:, :T]), "bf16", "extras fp8 gqa window: prefill")
    p = T
    for _ in range(3):
        check_close(m.decode_step(to_dev(toks[:, p])).cpu().numpy(), o.decode(toks[:, p]), "bf16",
                    "extras fp8 gqa window: decode")
        p += 1
    check_close(m.prefill(to_dev(toks[:, p:p + 30])).cpu().numpy(), o.extend(toks[:, p:p + 30]), "bf16",
                "extras fp8 gqa window: chunk")
    m.sync()
    m.close()
