"""Grouped-query attention and sliding-window layers on the GPU, through the C
ABI, against the fp64 oracle on the same seeded inputs (apidog.com/th "how
nanochat works" item 1: GQA with fewer K/V heads than query heads; a
configurable pattern such as "SSSL" of short and long attention windows).

Models at d12 widths (d_model 768, 6 query heads of 128) with 2, 3 or 6 K/V
heads (3, 2 or 1 query heads per K/V head: the odd group size exercises the
prefill attention's lone last head of a group), and "SL" patterns whose short
window cuts across 128-key blocks.  Tolerances: bf16 max 3e-2 / mean 5e-3,
fp32 1e-4.  The KV cache layout [layer][row][K/V head][position][dim] is
checked against the oracle's cached keys and values.
"""
import numpy as np
import pytest
import torch

import dense_gpt_transformer_fwd_b300 as ncp
import nc_inputs
from nc_testutil import check_close, oracle_for, small_bf16_shape, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gpt_transformer_fwd_b300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("n_kv,window,pattern", [(2, 0, ""), (3, 0, ""), (6, 0, ""), (3, 100, "SL"),
                                                 (1, 130, "LS"), (2, 64, "S")])
def test_prefill_and_decode(n_kv, window, pattern):
    sh = small_bf16_shape(n_layer=2, vocab=2048).with_(n_kv_head=n_kv, window=window, window_pattern=pattern)
    flat = nc_inputs.gen_weights(sh, 160 + n_kv)
    B, T, steps = 2, 300, 4
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 161)
    nxt = nc_inputs.gen_tokens(sh.vocab, (steps, B), 162)
    tag = f"gqa n_kv={n_kv} window={window}{pattern}"
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + steps + 40)
    check_close(m.prefill(to_dev(prompt)).cpu().numpy(), o.prefill(prompt), "bf16", f"{tag}: prefill")
    out = torch.empty((B, sh.vocab), device="cuda")
    for t in range(steps):
        got = m.decode_step(to_dev(nxt[t]), out=out).cpu().numpy()       # graph replay after step 1
        check_close(got, o.decode(nxt[t]), "bf16", f"{tag}: decode")
    chunk = nc_inputs.gen_tokens(sh.vocab, (B, 40), 163)
    check_close(m.prefill(to_dev(chunk)).cpu().numpy(), o.extend(chunk), "bf16", f"{tag}: chunk")
    m.sync()
    m.close()


def test_cache_layout_with_kv_heads():
    sh = small_bf16_shape(n_layer=2, vocab=512).with_(n_kv_head=3)
    flat = nc_inputs.gen_weights(sh, 164)
    B, T, maxb, maxs = 2, 40, 3, 48
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 165)
    o = oracle_for(flat, sh)
    o.prefill(prompt)
    m = ncp.Model(sh, flat, max_batch=maxb, max_seq=maxs)
    m.prefill(to_dev(prompt), last_only=True)
    k, v, guard, eb = m.kv_read()
    L, hd, nkv = sh.n_layer, sh.head_dim, sh.n_kv_head
    for raw, want in ((k, o.k_cache), (v, o.v_cache)):
        c = raw[guard:guard + L * maxb * nkv * maxs * hd].view(L, maxb, nkv, maxs, hd)
        for l in range(L):
            got = ((c[l, :B, :, :T].to(torch.int32) << 16).view(torch.float32)).cpu().numpy()
            np.testing.assert_allclose(got, want[l].transpose(0, 2, 1, 3), atol=2e-2, rtol=0)
        assert bool((c[:, :B, :, T:] == -1).all()) and bool((c[:, B:] == -1).all())
    m.close()


def test_long_context_window_decode():
    """Context 1500 with a 300-key window: the decode attention covers only
    the window's sub-chunks, split over a cluster of group CTAs per row."""
    sh = small_bf16_shape(n_layer=2, vocab=1024).with_(n_kv_head=3, window=300, window_pattern="SL")
    flat = nc_inputs.gen_weights(sh, 166)
    B, T, steps = 2, 1500, 3
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 167)
    nxt = nc_inputs.gen_tokens(sh.vocab, (steps, B), 168)
    o = oracle_for(flat, sh)
    o.prefill(prompt, logit_positions=[T - 1])
    m = ncp.Model(sh, flat, max_batch=B, max_seq=2048)
    m.prefill(to_dev(prompt), last_only=True)
    for t in range(steps):
        check_close(m.decode_step(to_dev(nxt[t])).cpu().numpy(), o.decode(nxt[t]), "bf16",
                    "gqa long-context window decode")
    m.sync()
    m.close()


def test_wide_batch_and_fp32_with_groups_and_windows():
    """136 rows (the generic one-position decode) with 3 K/V heads and a
    window; the fp32 model with 2 K/V heads (as many as query heads) and a
    window."""
    sh = small_bf16_shape(n_layer=2, vocab=1024).with_(n_kv_head=3, window=20, window_pattern="SL")
    flat = nc_inputs.gen_weights(sh, 169)
    B, T = 136, 33
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 170)
    nxt = nc_inputs.gen_tokens(sh.vocab, (2, B), 171)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + 2)
    check_close(m.prefill(to_dev(prompt), last_only=True).cpu().numpy(),
                o.prefill(prompt, logit_positions=[T - 1])[:, 0], "bf16", "gqa wide batch: prefill")
    for t in range(2):
        check_close(m.decode_step(to_dev(nxt[t])).cpu().numpy(), o.decode(nxt[t]), "bf16",
                    "gqa wide batch: decode")
    m.sync()
    m.close()
    tiny = nc_inputs.TINY.with_(n_kv_head=2, window=20, window_pattern="SL")
    flat = nc_inputs.gen_weights(tiny, 172)
    prompt = nc_inputs.gen_tokens(tiny.vocab, (2, 50), 173)
    nxt = nc_inputs.gen_tokens(tiny.vocab, (3, 2), 174)
    o = oracle_for(flat, tiny)
    m = ncp.Model(tiny, flat, max_batch=2, max_seq=53)
    check_close(m.prefill(to_dev(prompt)).cpu().numpy(), o.prefill(prompt), "f32", "gqa fp32: prefill")
    for t in range(3):
        check_close(m.decode_step(to_dev(nxt[t])).cpu().numpy(), o.decode(nxt[t]), "f32", "gqa fp32: decode")
    m.sync()
    m.close()
