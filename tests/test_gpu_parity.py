"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle
on the same seeded inputs.

Tolerances on logits: bf16 models max |dlogit| <= 3e-2 and mean <= 5e-3; the
fp32 model max <= 1e-4.  KV-cache indexing is checked bit-exactly (sentinels,
guards, unchanged rows, length).
"""
import numpy as np
import pytest
import torch

import dense_gpt_transformer_fwd_b300 as ncp
import nc_inputs
from nc_testutil import TOL, check_close, oracle_for, small_bf16_shape, to_dev, tokens_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gpt_transformer_fwd_b300 import build
    build.build()
    assert torch.cuda.is_available()


# ------------------------------------------------------------------ GEMM ---- #

@pytest.fixture(scope="module")
def small_model():
    sh = small_bf16_shape(n_layer=1, vocab=512)
    m = ncp.Model(sh, nc_inputs.gen_weights(sh, 5), max_batch=2, max_seq=64)
    yield m
    m.close()


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (64, 256, 128), (300, 512, 768),
                                   (1000, 1024, 1536), (257, 768, 3072), (2048, 4096, 768)])
def test_gemm_bf16_matches_fp32_matmul(small_model, M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    W = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), device="cuda")
    small_model.gemm_bf16(A, W, C)
    small_model.sync()
    ref = A.float() @ W.float().T
    err = (C - ref).abs().max().item()
    assert err <= 1e-4 * K ** 0.5 * 4, err


# ---------------------------------------------------------- tiny fp32 ---- #

def test_tiny_fp32_prefill_and_decode():
    w = nc_inputs.WORKLOADS["tiny"]
    flat = nc_inputs.gen_weights(w.shape, w.weight_seed)
    prompt, nxt = tokens_for(w)
    o = oracle_for(flat, w.shape)
    m = ncp.Model(w.shape, flat, max_batch=w.batch, max_seq=w.max_seq)
    got = m.prefill(to_dev(prompt)).cpu().numpy()
    check_close(got, o.prefill(prompt), "f32", "tiny prefill")
    for t in range(w.decode_steps):
        got = m.decode_step(to_dev(nxt[t])).cpu().numpy()
        check_close(got, o.decode(nxt[t]), "f32", f"tiny decode {t}")
    m.sync()
    assert m.kv_length() == (w.max_seq, w.batch)
    m.close()


# ------------------------------------------------------- small bf16 model --- #

@pytest.mark.parametrize("B,T,steps", [(3, 131, 5), (1, 1, 3), (2, 256, 2)])
def test_small_bf16_prefill_decode(B, T, steps):
    sh = small_bf16_shape()
    flat = nc_inputs.gen_weights(sh, 17)
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 18)
    nxt = nc_inputs.gen_tokens(sh.vocab, (steps, B), 19)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + steps)
    check_close(m.prefill(to_dev(prompt)).cpu().numpy(), o.prefill(prompt), "bf16", "prefill")
    for t in range(steps):
        check_close(m.decode_step(to_dev(nxt[t])).cpu().numpy(), o.decode(nxt[t]), "bf16",
                    f"decode {t}")
    m.sync()
    m.close()


@pytest.mark.parametrize("n_kv", [1, 3])
def test_persistent_prefill_attention_several_items_per_cta(n_kv):
    """More attention work items than SMs: 40 rows x 2 query tiles x 3 head
    pairs = 240 items on 148 persistent CTAs, so most CTAs run a second item
    of a different length (one or two key blocks), reloading the queries while
    the K/V ring continues; T = 200 leaves a ragged last query tile.  Every
    position of every row against the oracle, with one and with three K/V
    heads."""
    sh = small_bf16_shape(n_layer=2, vocab=512).with_(n_kv_head=n_kv)
    flat = nc_inputs.gen_weights(sh, 151 + n_kv)
    B, T = 40, 200
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 153)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T)
    got = m.prefill(to_dev(prompt)).cpu().numpy()
    check_close(got, oracle_for(flat, sh).prefill(prompt), "bf16", f"persistent attention, 240 items (n_kv={n_kv})")
    m.sync()
    m.close()


@pytest.mark.parametrize("B,T,steps", [(5, 130, 6), (40, 64, 4), (100, 33, 3)])
def test_decode_graph_replay_matches_oracle_and_eager(B, T, steps):
    """Decode steps into one fixed logits buffer are captured as a CUDA graph
    after the first step and replayed; they must match the oracle and be
    bit-identical to the eager steps of a second model (fresh buffer per step).
    B = 5, 40, 100 exercise the 32-, 64- and 128-column skinny GEMMs."""
    sh = small_bf16_shape(n_layer=2, vocab=2048)
    flat = nc_inputs.gen_weights(sh, 61)
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 62)
    nxt = nc_inputs.gen_tokens(sh.vocab, (steps, B), 63)
    o = oracle_for(flat, sh)
    o.prefill(prompt, logit_positions=[T - 1])
    g = ncp.Model(sh, flat, max_batch=B, max_seq=T + steps)
    e = ncp.Model(sh, flat, max_batch=B, max_seq=T + steps)
    g.prefill(to_dev(prompt), last_only=True)
    e.prefill(to_dev(prompt), last_only=True)
    out = torch.full((B, sh.vocab), float("nan"), device="cuda")
    for t in range(steps):
        tok = to_dev(nxt[t])
        got = g.decode_step(tok, out=out).cpu().numpy()
        ref = e.decode_step(tok).cpu().numpy()
        np.testing.assert_array_equal(got, ref)
        check_close(got, o.decode(nxt[t]), "bf16", f"graph decode step {t}")
    g.sync()
    e.sync()
    assert g.kv_length() == e.kv_length() == (T + steps, B)
    g.close()
    e.close()


def test_decode_attention_cluster_of_eight_groups():
    """Small batch, long context: the decode attention splits each row over a
    cluster of 8 group CTAs (max_seq 2048 -> 16 sub-chunks of 128 keys, 2 per
    group); at context 1501..1503 groups 6 and 7 hold no keys and only take part
    in the cluster barriers.  Graph-replayed steps match the oracle and the
    eager steps of a second model bit for bit."""
    sh = small_bf16_shape(n_layer=2, vocab=2048)
    flat = nc_inputs.gen_weights(sh, 71)
    B, T, steps, S = 2, 1500, 3, 2048
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 72)
    nxt = nc_inputs.gen_tokens(sh.vocab, (steps, B), 73)
    o = oracle_for(flat, sh)
    o.prefill(prompt, logit_positions=[T - 1])
    g = ncp.Model(sh, flat, max_batch=B, max_seq=S)
    e = ncp.Model(sh, flat, max_batch=B, max_seq=S)
    g.prefill(to_dev(prompt), last_only=True)
    e.prefill(to_dev(prompt), last_only=True)
    out = torch.full((B, sh.vocab), float("nan"), device="cuda")
    for t in range(steps):
        tok = to_dev(nxt[t])
        got = g.decode_step(tok, out=out).cpu().numpy()
        ref = e.decode_step(tok).cpu().numpy()
        np.testing.assert_array_equal(got, ref)
        check_close(got, o.decode(nxt[t]), "bf16", f"clustered decode step {t}")
    g.sync()
    e.sync()
    assert g.kv_length() == e.kv_length() == (T + steps, B)
    g.close()
    e.close()


def test_decode_attention_ragged_long_rows():
    """Rows of very different lengths (1 .. 1500 keys at B = 40) in one decode
    graph: each row's cluster of group CTAs covers its own context, so groups
    past a short row's keys hold nothing and long rows use every group.
    Sampled rows (the longest, the one-key row, a row of 129 keys and others)
    against their one-row oracles."""
    sh = small_bf16_shape(n_layer=2, vocab=2048)
    flat = nc_inputs.gen_weights(sh, 146)
    rng = np.random.default_rng(147)
    B, T, steps = 40, 1500, 3
    lens = rng.integers(1, T + 1, size=B)
    lens[0], lens[1], lens[-1] = T, 1, 129
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 148)
    nxt = nc_inputs.gen_tokens(sh.vocab, (steps, B), 149)
    rows = [0, 1, 7, 20, B - 1]
    orc = {b: oracle_for(flat, sh) for b in rows}
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + steps)
    m.prefill_rows(to_dev(prompt), lens, last_only=True)
    for b in rows:
        orc[b].prefill(prompt[b:b + 1, :lens[b]], logit_positions=[lens[b] - 1])
    out = torch.empty((B, sh.vocab), device="cuda")
    for t in range(steps):
        got = m.decode_step(to_dev(nxt[t]), out=out).cpu().numpy()
        for b in rows:
            check_close(got[b], orc[b].decode(nxt[t][b:b + 1])[0], "bf16", "decode attention, ragged long rows")
    m.sync()
    assert m.row_lengths() == (lens + steps).tolist()
    m.close()


def test_small_bf16_last_only_and_host_buffers():
    sh = small_bf16_shape()
    flat = nc_inputs.gen_weights(sh, 23)
    prompt = nc_inputs.gen_tokens(sh.vocab, (2, 77), 24)
    m = ncp.Model(sh, flat, max_batch=2, max_seq=80)
    full = m.prefill(to_dev(prompt)).cpu().numpy()
    m.kv_reset()
    last = m.prefill(to_dev(prompt), last_only=True).cpu().numpy()
    np.testing.assert_array_equal(last, full[:, -1])
    m.kv_reset()
    host = m.prefill(torch.from_numpy(prompt))            # host tokens, host (pinned) logits
    assert not host.is_cuda
    np.testing.assert_array_equal(host.numpy(), full)     # deterministic kernels
    m.sync()
    m.close()


# ------------------------------------------------------ KV-cache indexing --- #

def _cache_views(m, sh, max_batch, max_seq):
    k, v, guard, eb = m.kv_read()
    L, hd = sh.n_layer, sh.head_dim
    body = lambda t: t[guard:guard + L * max_batch * max_seq * hd].view(L, max_batch, max_seq, hd)
    return k, v, guard, body


def _as_float(t, eb):
    if eb == 2:
        return (t.to(torch.int32) << 16).view(torch.float32)  # bf16 bits -> fp32
    return t.view(torch.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_kv_cache_indexing_bit_exact(dtype):
    if dtype == "bf16":
        sh, B, T, steps, maxb, maxs = small_bf16_shape(), 2, 40, 3, 3, 48
    else:
        sh, B, T, steps, maxb, maxs = nc_inputs.TINY, 2, 20, 3, 3, 30
    flat = nc_inputs.gen_weights(sh, 31)
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 32)
    nxt = nc_inputs.gen_tokens(sh.vocab, (steps, B), 33)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=maxb, max_seq=maxs)
    k0, v0, guard, _ = _cache_views(m, sh, maxb, maxs)
    sentinel = -1                                        # every byte 0xFF
    assert bool((k0 == sentinel).all()) and bool((v0 == sentinel).all())
    m.prefill(to_dev(prompt))
    o.prefill(prompt)
    snaps = []
    for t in range(steps + 1):
        m.sync()
        n = T + t
        assert m.kv_length() == (n, B)
        k, v, guard, body = _cache_views(m, sh, maxb, maxs)
        eb = 2 if dtype == "bf16" else 4
        for raw in (k, v):
            assert bool((raw[:guard] == sentinel).all()) and bool((raw[-guard:] == sentinel).all())
            c = body(raw)
            assert bool((c[:, B:] == sentinel).all())            # rows beyond the batch
            assert bool((c[:, :B, n:] == sentinel).all())        # positions beyond the length
        for l in range(sh.n_layer):
            gk = _as_float(body(k)[l, :B, :n], eb).cpu().numpy()
            gv = _as_float(body(v)[l, :B, :n], eb).cpu().numpy()
            tol = 2e-2 if dtype == "bf16" else 1e-5
            np.testing.assert_allclose(gk, o.k_cache[l][:, :, 0, :], atol=tol, rtol=0)
            np.testing.assert_allclose(gv, o.v_cache[l][:, :, 0, :], atol=tol, rtol=0)
        snaps.append((body(k)[:, :B, :n].clone(), body(v)[:, :B, :n].clone()))
        for (sk, sv) in snaps[:-1]:                                # earlier rows never rewritten
            p = sk.shape[2]
            assert torch.equal(body(k)[:, :B, :p], sk) and torch.equal(body(v)[:, :B, :p], sv)
        if t < steps:
            m.decode_step(to_dev(nxt[t]))
            o.decode(nxt[t])
    m.close()


# ------------------------------------------------------------ error paths --- #

def test_state_and_capacity_errors():
    sh = small_bf16_shape(n_layer=1, vocab=512)
    m = ncp.Model(sh, nc_inputs.gen_weights(sh, 41), max_batch=2, max_seq=9)
    tok = to_dev(nc_inputs.gen_tokens(sh.vocab, (2, 8), 42))
    with pytest.raises(ncp.NcError) as e:
        m.decode_step(tok[:, 0])
    assert e.value.name == "NC_ERR_STATE"
    m.prefill(tok)
    with pytest.raises(ncp.NcError) as e:           # a second chunk of 8 would pass max_seq
        m.prefill(tok)
    assert e.value.name == "NC_ERR_CAPACITY"
    with pytest.raises(ncp.NcError) as e:
        m.decode_step(tok[:1, 0])
    assert e.value.name == "NC_ERR_INVALID_ARG"
    m.decode_step(tok[:, 0])                         # length 8 -> 9 == max_seq
    with pytest.raises(ncp.NcError) as e:
        m.decode_step(tok[:, 1])
    assert e.value.name == "NC_ERR_CAPACITY"
    m.kv_reset()
    with pytest.raises(ncp.NcError) as e:
        m.prefill(to_dev(np.zeros((3, 4), np.int32)))
    assert e.value.name == "NC_ERR_INVALID_ARG"
    with pytest.raises(ncp.NcError):
        m.prefill(to_dev(np.zeros((1, 10), np.int32)))
    m.sync()
    m.close()


def test_oom_reported_and_context_survives():
    """A cache larger than the device (2^18 rows x 8192 positions x 128 bf16 =
    512 GiB per tensor, the first large allocation) fails with NC_ERR_OOM,
    frees what was allocated, and the next model still computes."""
    sh = small_bf16_shape(n_layer=1, vocab=512)
    w = nc_inputs.gen_weights(sh, 44)
    free0 = torch.cuda.mem_get_info()[0]
    with pytest.raises(ncp.NcError) as e:
        ncp.Model(sh, w, max_batch=1 << 18, max_seq=8192)
    assert e.value.name == "NC_ERR_OOM"
    assert "memory" in str(e.value)
    assert torch.cuda.mem_get_info()[0] >= free0 - (64 << 20)
    tok = nc_inputs.gen_tokens(sh.vocab, (1, 12), 45)
    m = ncp.Model(sh, w, max_batch=1, max_seq=12)
    check_close(m.prefill(to_dev(tok)).cpu().numpy(), oracle_for(w, sh).prefill(tok), "bf16", "after OOM")
    m.close()


def test_bad_token_reported_by_sync():
    sh = small_bf16_shape(n_layer=1, vocab=512)
    m = ncp.Model(sh, nc_inputs.gen_weights(sh, 43), max_batch=1, max_seq=8)
    tok = np.array([[1, 2, 512, 3]], np.int32)
    m.prefill(to_dev(tok))
    assert ncp.nc.STATUS[m.sync_status()] == "NC_ERR_TOKEN"
    assert m.sync_status() == 0                      # the error word is cleared
    m.close()


def test_bounded_wait_times_out_and_context_survives():
    sh = small_bf16_shape(n_layer=1, vocab=512)
    flat = nc_inputs.gen_weights(sh, 44)
    m = ncp.Model(sh, flat, max_batch=1, max_seq=8)
    m.debug_wait_timeout(20_000_000)                 # 20 ms on an mbarrier nothing arrives at
    assert ncp.nc.STATUS[m.sync_status()] == "NC_ERR_TIMEOUT"
    tok = nc_inputs.gen_tokens(sh.vocab, (1, 8), 45)
    got = m.prefill(to_dev(tok)).cpu().numpy()       # the context is still usable
    m.sync()
    check_close(got, oracle_for(flat, sh).prefill(tok), "bf16", "after timeout")
    m.close()


# ------------------------------------------------- full-size workloads ---- #

def test_d12_prefill_full_size_sampled_rows():
    """8 x 2048 prefill of d12 in the benchmark's launch configuration; the
    oracle recomputes rows 0 and 7 (rows are independent) at every position."""
    w = nc_inputs.WORKLOADS["d12_prefill"]
    flat = nc_inputs.gen_weights(w.shape, w.weight_seed)
    prompt, _ = tokens_for(w)
    m = ncp.Model(w.shape, flat, max_batch=w.batch, max_seq=w.max_seq)
    got = m.prefill(to_dev(prompt))
    m.sync()
    rows = [0, w.batch - 1]
    sample = got[rows].cpu().numpy()
    assert np.all(np.isfinite(got.cpu().numpy()))
    m.close()
    del got
    want = oracle_for(flat, w.shape).prefill(prompt[rows])
    check_close(sample, want, "bf16", "d12 prefill rows 0, 7")


def test_d12_decode_full_size_sampled_rows():
    """32 x 512 prompt + 256 decode steps of d12; rows 0, 15, 31 checked at every step."""
    w = nc_inputs.WORKLOADS["d12_decode"]
    flat = nc_inputs.gen_weights(w.shape, w.weight_seed)
    prompt, nxt = tokens_for(w)
    rows = [0, 15, 31]
    m = ncp.Model(w.shape, flat, max_batch=w.batch, max_seq=w.max_seq)
    m.prefill(to_dev(prompt), last_only=True)
    got = []
    for t in range(w.decode_steps):
        got.append(m.decode_step(to_dev(nxt[t]))[rows].cpu().numpy())
    m.sync()
    assert m.kv_length() == (w.max_seq, w.batch)
    m.close()
    o = oracle_for(flat, w.shape)
    o.prefill(prompt[rows], logit_positions=[w.prompt_len - 1])
    for t in range(w.decode_steps):
        check_close(got[t], o.decode(nxt[t][rows]), "bf16", f"d12 decode step {t}")
