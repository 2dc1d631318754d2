"""nc_decode_step_noalloc: the decode step for callers that must not allocate
device memory while they decode (a serving loop that has given every free
byte to other models' KV caches, or a host framework that owns the allocator).
Every intermediate lives in model-owned buffers sized at creation and the
step runs kernel by kernel (no graph instantiation).

Checked here against nc_decode_step, through the C ABI, on two calls in a row,
within the bf16 logit tolerance the other tests use.  This file is collected
last so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

import dense_gpt_transformer_fwd_b300 as ncp
import nc_inputs
from nc_testutil import check_close, small_bf16_shape, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gpt_transformer_fwd_b300 import build
    build.build()
    assert torch.cuda.is_available()


def test_noalloc_decode_matches_decode_step_two_calls():
    sh = small_bf16_shape(n_layer=2, vocab=4096)
    flat = nc_inputs.gen_weights(sh, 91)
    B, T = 3, 300                                   # context 301, 302: three 128-key chunks
    prompt = to_dev(nc_inputs.gen_tokens(sh.vocab, (B, T), 92))
    nxt = to_dev(nc_inputs.gen_tokens(sh.vocab, (2, B), 93))
    ref = ncp.Model(sh, flat, max_batch=B, max_seq=T + 2)
    dut = ncp.Model(sh, flat, max_batch=B, max_seq=T + 2)
    ref.prefill(prompt, last_only=True)
    dut.prefill(prompt, last_only=True)
    out = torch.full((B, sh.vocab), float("nan"), device="cuda")
    for t in range(2):
        want = ref.decode_step(nxt[t]).cpu().numpy()
        got = dut.decode_step_noalloc(nxt[t], out).cpu().numpy()
        ref.sync()
        dut.sync()
        check_close(got, want, "bf16", f"no-alloc decode call {t}")
        assert dut.kv_length() == ref.kv_length() == (T + t + 1, B)
    ref.close()
    dut.close()


def test_noalloc_decode_rejects_host_buffers_and_runs_long_contexts():
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
