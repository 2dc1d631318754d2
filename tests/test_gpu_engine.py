"""The engine steps around the forward pass on the GPU, through the C ABI,
against the fp64 oracle on the same seeded inputs (apidog.com/th "how
nanochat works" item 6: KV cache, prefill and decode, batch generation that
clones the cache for parallel sampling):

* chunked prefill: a prompt prefilled in chunks, with decode steps between
  chunks, against the oracle's prefill / extend / decode;
* KV-cache clone: one row's cache copied to n rows, then n different
  continuations, against the oracle's clone_row;
* sampling: next tokens on the device against the oracle's sample_tokens,
  bit-exact (token ids are integers; both sides decide in fp64), with planted
  ties for the greedy rule and at the top-k threshold;
* the generation loop decode -> sample -> decode with device tokens only.

Logit tolerances: bf16 max 3e-2 / mean 5e-3, fp32 1e-4.
"""
import numpy as np
import pytest
import torch

import dense_gpt_transformer_fwd_b300 as ncp
import nc_inputs
from nc_testutil import check_close, oracle_for, small_bf16_shape, to_dev
from oracle.gpt_oracle import sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gpt_transformer_fwd_b300 import build
    build.build()
    assert torch.cuda.is_available()


# ------------------------------------------------------------ chunked prefill

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chunked_prefill_with_decode_between_chunks(dtype):
    """Chunks of 150 and 90 positions (the second starts off a 128-key block
    boundary), two decode steps, a third chunk of 70 (its attention reads
    keys written by decode steps), one more decode step."""
    if dtype == "bf16":
        sh = small_bf16_shape(n_layer=2, vocab=2048)
    else:
        sh = nc_inputs.TINY
    flat = nc_inputs.gen_weights(sh, 111)
    B = 2
    chunks = [150, 90]
    total = sum(chunks) + 2 + 70 + 1
    toks = nc_inputs.gen_tokens(sh.vocab, (B, total), 112)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=total)
    p = 0
    got = m.prefill(to_dev(toks[:, :150])).cpu().numpy()
    check_close(got, o.prefill(toks[:, :150]), dtype, "chunked prefill: chunk 1")
    p = 150
    got = m.prefill(to_dev(toks[:, p:p + 90])).cpu().numpy()
    check_close(got, o.extend(toks[:, p:p + 90]), dtype, "chunked prefill: chunk 2 at 150")
    p += 90
    for t in range(2):
        got = m.decode_step(to_dev(toks[:, p])).cpu().numpy()
        check_close(got, o.decode(toks[:, p]), dtype, "chunked prefill: decode between chunks")
        p += 1
    got = m.prefill(to_dev(toks[:, p:p + 70]), last_only=True).cpu().numpy()
    check_close(got, o.extend(toks[:, p:p + 70], logit_positions=[69])[:, 0], dtype,
                "chunked prefill: chunk 3 after decode (last position)")
    p += 70
    got = m.decode_step(to_dev(toks[:, p])).cpu().numpy()
    check_close(got, o.decode(toks[:, p]), dtype, "chunked prefill: decode after chunk 3")
    m.sync()
    assert m.kv_length() == (total, B)
    m.close()


def test_chunked_prefill_equals_whole_prefill_and_capacity():
    sh = small_bf16_shape(n_layer=2, vocab=2048)
    flat = nc_inputs.gen_weights(sh, 113)
    B, T = 3, 384
    toks = nc_inputs.gen_tokens(sh.vocab, (B, T), 114)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T)
    whole = m.prefill(to_dev(toks)).cpu().numpy()
    m.kv_reset()
    parts = []
    for a, b in ((0, 128), (128, 129), (129, 300), (300, 384)):   # 128, 1, 171, 84 positions
        parts.append(m.prefill(to_dev(toks[:, a:b])).cpu().numpy())
    m.sync()
    check_close(np.concatenate(parts, axis=1), whole, "bf16", "chunked vs whole prefill")
    assert m.kv_length() == (T, B)
    with pytest.raises(ncp.NcError) as e:                 # the cache is full
        m.prefill(to_dev(toks[:, :1]))
    assert e.value.name == "NC_ERR_CAPACITY"
    m.kv_reset()
    m.prefill(to_dev(toks[:, :10]))
    with pytest.raises(ncp.NcError) as e:                 # a chunk must keep the batch
        m.prefill(to_dev(toks[:2, 10:20]))
    assert e.value.name == "NC_ERR_INVALID_ARG"
    m.sync()
    m.close()


# -------------------------------------------------------------- cache clone

def test_kv_clone_then_parallel_continuations():
    """Prefill one prompt (B = 1), clone its cache to 5 rows, decode 3 steps
    with a different token per row; then a chunk of 40 positions per row."""
    sh = small_bf16_shape(n_layer=2, vocab=2048)
    flat = nc_inputs.gen_weights(sh, 115)
    n, T = 5, 100
    prompt = nc_inputs.gen_tokens(sh.vocab, (1, T), 116)
    nxt = nc_inputs.gen_tokens(sh.vocab, (3, n), 117)
    chunk = nc_inputs.gen_tokens(sh.vocab, (n, 40), 118)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=n, max_seq=T + 3 + 40)
    check_close(m.prefill(to_dev(prompt), last_only=True).cpu().numpy(),
                o.prefill(prompt, logit_positions=[T - 1])[:, 0], "bf16", "clone: prompt")
    m.kv_clone(0, n)
    o.clone_row(0, n)
    assert m.kv_length() == (T, n)
    for t in range(3):
        check_close(m.decode_step(to_dev(nxt[t])).cpu().numpy(), o.decode(nxt[t]), "bf16",
                    "clone: decode of the cloned rows")
    check_close(m.prefill(to_dev(chunk)).cpu().numpy(), o.extend(chunk), "bf16", "clone: chunk after decode")
    m.sync()
    with pytest.raises(ncp.NcError) as e:
        m.kv_clone(n, 2)                                   # src must be a cached row
    assert e.value.name == "NC_ERR_INVALID_ARG"
    m.close()


def test_kv_clone_copies_rows_bit_exactly():
    sh = small_bf16_shape(n_layer=2, vocab=512)
    flat = nc_inputs.gen_weights(sh, 119)
    m = ncp.Model(sh, flat, max_batch=4, max_seq=64)
    m.prefill(to_dev(nc_inputs.gen_tokens(sh.vocab, (3, 50), 120)), last_only=True)
    m.kv_clone(1, 4)
    k, v, guard, eb = m.kv_read()
    L, hd = sh.n_layer, sh.head_dim
    for raw in (k, v):
        c = raw[guard:guard + L * 4 * 64 * hd].view(L, 4, 64, hd)
        for b in range(4):
            assert torch.equal(c[:, b, :50], c[:, 1, :50])
        assert bool((c[:, 3, 50:] == -1).all())           # row 3 beyond the length keeps the sentinel
    m.close()


# ----------------------------------------------------------------- sampling

def _planted_logits(B, V, seed):
    """Seeded logits with planted ties: row 0 has three equal maxima, row 1
    is quantised to steps of 0.25 (many ties at every threshold), row 2 is
    constant, the rest are normal draws times 3."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((B, V)) * 3.0).astype(np.float32)
    x[0, [7, 100, V - 3]] = x[0].max() + 1.0
    if B > 1:
        x[1] = np.round(x[1] * 4.0) / 4.0
    if B > 2:
        x[2] = 0.5
    return x


@pytest.mark.parametrize("temperature,top_k", [(0.0, 0), (1.0, 1), (1.0, 5), (0.7, 50), (1.5, 50),
                                               (1.0, 1000), (2.0, 1024)])
def test_sampling_matches_oracle_bit_exactly(temperature, top_k):
    sh = small_bf16_shape(n_layer=1, vocab=4096)
    B, V = 12, sh.vocab
    m = ncp.Model(sh, nc_inputs.gen_weights(sh, 121), max_batch=B, max_seq=8)
    logits = _planted_logits(B, V, 122)
    u = np.random.default_rng(123).random(B)
    got = m.sample(to_dev(logits), temperature, top_k, to_dev(u)).cpu().numpy()
    m.sync()
    want = sample_tokens(logits.astype(np.float64), temperature, top_k, u)
    np.testing.assert_array_equal(got, want)
    if temperature == 0.0:
        assert got[0] == 7 and got[2] == 0                  # lowest index among equal maxima
    m.close()


@pytest.mark.parametrize("temperature,top_k", [(0.0, 0), (0.8, 50), (1.0, 1024)])
def test_sampling_full_vocabulary_bit_exactly(temperature, top_k):
    """The sampling kernel over the workloads' 65,536-token vocabulary (its
    radix select ranks 16x more candidates than in the test above), on the
    same kind of seeded logits with planted ties."""
    sh = small_bf16_shape(n_layer=1, vocab=65536)
    B, V = 8, sh.vocab
    m = ncp.Model(sh, nc_inputs.gen_weights(sh, 131), max_batch=B, max_seq=8)
    logits = _planted_logits(B, V, 132)
    u = np.random.default_rng(133).random(B)
    got = m.sample(to_dev(logits), temperature, top_k, to_dev(u)).cpu().numpy()
    m.sync()
    np.testing.assert_array_equal(got, sample_tokens(logits.astype(np.float64), temperature, top_k, u))
    m.close()


def test_sampling_whole_vocabulary_and_limits():
    """top_k = 0 keeps every candidate: on the device only while the
    vocabulary has at most 1024 entries (the tiny model's 512); otherwise the
    call is refused."""
    tiny = nc_inputs.TINY
    B = 6
    m = ncp.Model(tiny, nc_inputs.gen_weights(tiny, 124), max_batch=B, max_seq=8)
    logits = _planted_logits(B, tiny.vocab, 125)
    for seed, temp in ((126, 1.0), (127, 0.3), (128, 4.0)):
        u = np.random.default_rng(seed).random(B)
        got = m.sample(to_dev(logits), temp, 0, to_dev(u)).cpu().numpy()
        np.testing.assert_array_equal(got, sample_tokens(logits.astype(np.float64), temp, 0, u))
    m.close()
    sh = small_bf16_shape(n_layer=1, vocab=4096)
    m = ncp.Model(sh, nc_inputs.gen_weights(sh, 129), max_batch=2, max_seq=8)
    lg = to_dev(_planted_logits(2, sh.vocab, 130))
    u = to_dev(np.array([0.1, 0.9]))
    for top_k in (0, 1025):
        with pytest.raises(ncp.NcError) as e:
            m.sample(lg, 1.0, top_k, u)
        assert e.value.name == "NC_ERR_UNSUPPORTED"
    with pytest.raises(ncp.NcError) as e:
        m.sample(lg, -1.0, 5, u)
    assert e.value.name == "NC_ERR_INVALID_ARG"
    m.close()


def test_generation_loop_on_device():
    """Prefill one prompt, clone it to 4 rows, then 6 steps of decode ->
    sample (temperature 1, top_k 50, a different draw per row) -> decode, the
    tokens never leaving the device.  Each sampled token equals the oracle's
    sample_tokens on the GPU's logits and draws; the GPU's logits match the
    oracle fed the same tokens."""
    sh = small_bf16_shape(n_layer=2, vocab=2048)
    flat = nc_inputs.gen_weights(sh, 131)
    n, T, steps = 4, 64, 6
    prompt = nc_inputs.gen_tokens(sh.vocab, (1, T), 132)
    draws = np.random.default_rng(133).random((steps, n))
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=n, max_seq=T + steps + 1)
    first = m.prefill(to_dev(prompt), last_only=True)
    o.prefill(prompt, logit_positions=[T - 1])
    m.kv_clone(0, n)
    o.clone_row(0, n)
    u_d = to_dev(draws)
    tok = m.sample(first.expand(n, -1).contiguous(), 1.0, 50, u_d[0])
    logits = torch.empty((n, sh.vocab), device="cuda")
    for t in range(steps):
        tok_h = tok.cpu().numpy()
        m.decode_step(tok, out=logits)
        lg = logits.cpu().numpy()
        check_close(lg, o.decode(tok_h), "bf16", "generation loop: logits")
        if t + 1 < steps:
            tok = m.sample(logits, 1.0, 50, u_d[t + 1])
            np.testing.assert_array_equal(tok.cpu().numpy(),
                                          sample_tokens(lg.astype(np.float64), 1.0, 50, draws[t + 1]))
    m.sync()
    assert m.kv_length() == (T + steps, n)
    m.close()


# --------------------------------------------------------- per-row lengths

@pytest.mark.parametrize("dtype,B", [("bf16", 4), ("bf16", 136), ("f32", 3)])
def test_rows_of_different_lengths(dtype, B):
    """Prompts of different lengths in one padded prefill, decode steps at
    each row's own position (through the decode graph: one fixed logits
    buffer), a ragged second chunk, more decode steps, then a clone of one
    row to all rows.  Rows are independent, so each is checked against its
    own one-row oracle.  B = 136 is wider than the decode GEMMs (the generic
    one-position pass)."""
    sh = small_bf16_shape(n_layer=2, vocab=2048) if dtype == "bf16" else nc_inputs.TINY
    flat = nc_inputs.gen_weights(sh, 141)
    rng = np.random.default_rng(142)
    T1, T2 = 130, 64
    lens1 = rng.integers(1, T1 + 1, size=B)
    lens1[0], lens1[-1] = T1, 1
    lens2 = rng.integers(1, T2 + 1, size=B)
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T1), 143)
    chunk = nc_inputs.gen_tokens(sh.vocab, (B, T2), 144)
    nxt = nc_inputs.gen_tokens(sh.vocab, (6, B), 145)
    orc = [oracle_for(flat, sh) for _ in range(B)]
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T1 + 3 + T2 + 2 + 1)
    got = m.prefill_rows(to_dev(prompt), lens1).cpu().numpy()
    for b in range(B):
        check_close(got[b, :lens1[b]], orc[b].prefill(prompt[b:b + 1, :lens1[b]])[0], dtype,
                    f"ragged rows (B={B}): prefill")
    assert m.row_lengths() == lens1.tolist()
    out = torch.empty((B, sh.vocab), device="cuda")
    step = 0

    def decode_all(what):
        nonlocal step
        got = m.decode_step(to_dev(nxt[step]), out=out).cpu().numpy()
        for b in range(B):
            check_close(got[b], orc[b].decode(nxt[step][b:b + 1])[0], dtype, f"ragged rows (B={B}): {what}")
        step += 1

    for _ in range(3):
        decode_all("decode")
    got = m.prefill_rows(to_dev(chunk), lens2, last_only=True).cpu().numpy()
    for b in range(B):
        want = orc[b].extend(chunk[b:b + 1, :lens2[b]], logit_positions=[lens2[b] - 1])[0, 0]
        check_close(got[b], want, dtype, f"ragged rows (B={B}): second chunk, last token")
    for _ in range(2):
        decode_all("decode after the chunk")
    assert m.row_lengths() == (lens1 + 3 + lens2 + 2).tolist()
    src = B // 2
    m.kv_clone(src, B)
    assert m.row_lengths() == [int(lens1[src] + 3 + lens2[src] + 2)] * B
    o = orc[src]
    o.clone_row(0, B)
    got = m.decode_step(to_dev(nxt[5])).cpu().numpy()
    check_close(got, o.decode(nxt[5]), dtype, f"ragged rows (B={B}): decode after a clone")
    m.sync()
    m.close()
