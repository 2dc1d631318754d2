"""FP8 projection weights on the GPU, through the C ABI, against the fp64
oracle on the same seeded inputs (the FP8 path of apidog.com/th "how nanochat
works" item 3, used here for inference).

The weights of an fp8 model are rounded by the shared input generators to
E4M3 values times one power-of-two scale per matrix; the oracle consumes
exactly those values.  On the GPU the decode GEMMs stream the E4M3 bytes and
widen them exactly to f16 (f16 activations), and the prefill runs on the
exact bf16 image of the same weights, so the bf16 tolerances apply: max
|dlogit| <= 3e-2, mean <= 5e-3.
"""
import numpy as np
import pytest
import torch

import dense_gpt_transformer_fwd_b300 as ncp
import nc_inputs
from nc_testutil import check_close, oracle_for, small_bf16_shape, to_dev, tokens_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gpt_transformer_fwd_b300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("B,n_kv", [(5, 1), (40, 1), (100, 1), (6, 3)])
def test_fp8_prefill_and_decode(B, n_kv):
    """B = 5, 40, 100: the 32-, 64- and 128-column FP8 decode GEMMs (graph
    replay after the first step); 3 K/V heads at B = 6."""
    sh = small_bf16_shape(n_layer=2, vocab=2048).with_(dtype="fp8", n_kv_head=n_kv)
    flat = nc_inputs.gen_weights(sh, 180 + B)
    T, steps = 70, 4
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 181)
    nxt = nc_inputs.gen_tokens(sh.vocab, (steps, B), 182)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + steps)
    check_close(m.prefill(to_dev(prompt), last_only=True).cpu().numpy(),
                o.prefill(prompt, logit_positions=[T - 1])[:, 0], "bf16", f"fp8 B={B}: prefill")
    out = torch.empty((B, sh.vocab), device="cuda")
    for t in range(steps):
        got = m.decode_step(to_dev(nxt[t]), out=out).cpu().numpy()
        check_close(got, o.decode(nxt[t]), "bf16", f"fp8 B={B}: decode")
    m.sync()
    m.close()


def test_fp8_noalloc_equals_decode_step():
    sh = small_bf16_shape(n_layer=2, vocab=2048).with_(dtype="fp8")
    flat = nc_inputs.gen_weights(sh, 190)
    B, T = 4, 50
    prompt = to_dev(nc_inputs.gen_tokens(sh.vocab, (B, T), 191))
    tok = to_dev(nc_inputs.gen_tokens(sh.vocab, (B,), 192))
    ref = ncp.Model(sh, flat, max_batch=B, max_seq=T + 1)
    dut = ncp.Model(sh, flat, max_batch=B, max_seq=T + 1)
    ref.prefill(prompt, last_only=True)
    dut.prefill(prompt, last_only=True)
    out = torch.empty((B, sh.vocab), device="cuda")
    want = ref.decode_step(tok).cpu().numpy()
    got = dut.decode_step_noalloc(tok, out).cpu().numpy()
    ref.sync()
    dut.sync()
    np.testing.assert_array_equal(got, want)
    ref.close()
    dut.close()


def test_fp8_d24_decode_full_size_sampled_rows():
    """The d24 decode workload with FP8 weights in the benchmark's launch
    configuration (128 rows, 2048-token prompt); rows 0, 64 and 127 checked at
    each of the first 16 steps."""
    w = nc_inputs.WORKLOADS["d24_decode_fp8"]
    flat = nc_inputs.gen_weights(w.shape, w.weight_seed)
    prompt, nxt = tokens_for(w)
    rows, steps = [0, w.batch // 2, w.batch - 1], 16
    m = ncp.Model(w.shape, flat, max_batch=w.batch, max_seq=w.max_seq)
    m.prefill(to_dev(prompt), last_only=True)
    out = torch.empty((w.batch, w.shape.vocab), device="cuda")
    nxt_d = to_dev(nxt)
    got = []
    for t in range(steps):
        m.decode_step(nxt_d[t], out=out)
        got.append(out[rows].cpu().numpy())
    m.sync()
    m.close()
    torch.cuda.empty_cache()
    o = oracle_for(flat, w.shape)
    o.prefill(prompt[rows], logit_positions=[w.prompt_len - 1])
    for t in range(steps):
        check_close(got[t], o.decode(nxt[t][rows]), "bf16", "d24_decode_fp8 step")
