"""nc_decode_step_noalloc: the decode step for callers that cannot allocate
device memory while they decode (a serving loop that has handed every free
byte to other models' KV caches, or a host framework that owns the device
allocator).  The step's intermediates live in a fixed scratch array that is
part of the library, resolved when a model is created; the call itself
allocates nothing and does no set-up.

Checked here, through the C ABI:
  * the first decode of a fresh model goes through this call, the device's
    free memory (cudaMemGetInfo) does not shrink across two calls, and the
    logits match the fp64 oracle;
  * two calls in a row match nc_decode_step on a twin model within the bf16
    logit tolerance the other tests use (max 3e-2, mean 5e-3), and the oracle;
  * host buffers, and batches or models beyond the scratch, are refused with
    nothing enqueued; a long context at 64 rows matches nc_decode_step.
This file is collected last so that a run stopping at the first failure has
run every other test.  It passes alone in a fresh process too.
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


def test_noalloc_first_decode_allocates_nothing_and_matches_oracle():
    sh = small_bf16_shape(n_layer=2, vocab=4096)
    flat = nc_inputs.gen_weights(sh, 97)
    B, T = 5, 140
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 98)
    nxt = nc_inputs.gen_tokens(sh.vocab, (2, B), 99)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + 2)
    tok = to_dev(nxt)
    last = torch.empty((B, sh.vocab), device="cuda")
    outs = [torch.full((B, sh.vocab), float("nan"), device="cuda") for _ in range(2)]
    m.prefill(to_dev(prompt), last_only=True, out=last)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for t in range(2):
        m.decode_step_noalloc(tok[t], outs[t])
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    m.sync()
    assert free1 >= free0, f"device free memory shrank by {free0 - free1} bytes"
    assert m.kv_length() == (T + 2, B)
    o = oracle_for(flat, sh)
    o.prefill(prompt, logit_positions=[T - 1])
    for t in range(2):
        check_close(outs[t].cpu().numpy(), o.decode(nxt[t]), "bf16", f"no-alloc decode vs oracle call {t}")
    m.close()


def test_noalloc_decode_matches_decode_step_two_calls():
    sh = small_bf16_shape(n_layer=2, vocab=4096)
    flat = nc_inputs.gen_weights(sh, 91)
    B, T = 3, 300                                   # context 301, 302: three 128-key chunks
    prompt_h = nc_inputs.gen_tokens(sh.vocab, (B, T), 92)
    nxt_h = nc_inputs.gen_tokens(sh.vocab, (2, B), 93)
    prompt, nxt = to_dev(prompt_h), to_dev(nxt_h)
    ref = ncp.Model(sh, flat, max_batch=B, max_seq=T + 2)
    dut = ncp.Model(sh, flat, max_batch=B, max_seq=T + 2)
    ref.prefill(prompt, last_only=True)
    dut.prefill(prompt, last_only=True)
    o = oracle_for(flat, sh)
    o.prefill(prompt_h, logit_positions=[T - 1])
    out = torch.full((B, sh.vocab), float("nan"), device="cuda")
    for t in range(2):
        want = ref.decode_step(nxt[t]).cpu().numpy()
        got = dut.decode_step_noalloc(nxt[t], out).cpu().numpy()
        ref.sync()
        dut.sync()
        check_close(got, want, "bf16", f"no-alloc decode vs nc_decode_step call {t}")
        check_close(got, o.decode(nxt_h[t]), "bf16", f"no-alloc decode vs oracle call {t}")
        assert dut.kv_length() == ref.kv_length() == (T + t + 1, B)
    ref.close()
    dut.close()


def test_noalloc_decode_refusals_and_long_context():
    """Host buffers are refused with nothing enqueued; a long context at a
    large batch (64 rows, 5121 keys, the attention split over a cluster of
    groups per row) matches nc_decode_step."""
    sh = small_bf16_shape(n_layer=1, vocab=512)
    flat = nc_inputs.gen_weights(sh, 94)
    B, T = 64, 5120
    prompt = to_dev(nc_inputs.gen_tokens(sh.vocab, (B, T), 95))
    tok = to_dev(nc_inputs.gen_tokens(sh.vocab, (B,), 96))
    ref = ncp.Model(sh, flat, max_batch=B, max_seq=T + 1)
    dut = ncp.Model(sh, flat, max_batch=B, max_seq=T + 1)
    ref.prefill(prompt, last_only=True)
    dut.prefill(prompt, last_only=True)
    out = torch.empty((B, sh.vocab), device="cuda")
    with pytest.raises(ncp.NcError) as e:
        dut.decode_step_noalloc(tok.cpu(), out)
    assert e.value.name == "NC_ERR_INVALID_ARG"
    assert dut.kv_length() == (T, B)                # nothing was enqueued
    want = ref.decode_step(tok).cpu().numpy()
    got = dut.decode_step_noalloc(tok, out).cpu().numpy()
    ref.sync()
    dut.sync()
    check_close(got, want, "bf16", "no-alloc decode at context 5121")
    assert dut.kv_length() == (T + 1, B)
    ref.close()
    dut.close()


@pytest.mark.parametrize("case", ["rows", "width"])
def test_noalloc_decode_beyond_the_scratch(case):
    """160 rows, or a model wider than the scratch (d_model 2304, d_mlp 9216),
    return NC_ERR_SCRATCH_LIMIT with nothing enqueued."""
    if case == "rows":
        sh, B = small_bf16_shape(n_layer=1, vocab=512), 160
    else:
        sh = nc_inputs.D12.with_(name="wide", n_layer=1, d_model=2304, n_head=16, d_mlp=9216, vocab=512)
        B = 2
    flat = nc_inputs.gen_weights(sh, 100)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=9)
    m.prefill(to_dev(nc_inputs.gen_tokens(sh.vocab, (B, 8), 101)), last_only=True)
    out = torch.empty((B, sh.vocab), device="cuda")
    with pytest.raises(ncp.NcError) as e:
        m.decode_step_noalloc(to_dev(np.zeros(B, np.int32)), out)
    assert e.value.name == "NC_ERR_SCRATCH_LIMIT"
    assert m.kv_length() == (8, B)
    m.sync()
    m.close()
