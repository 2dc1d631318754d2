"""Pins of the oracle's grouped-query attention (R12) and sliding-window
attention (R13), against what the pages and the mathematics fix:

* apidog.com/th "how nanochat works" item 1: grouped-query attention (fewer
  K/V heads than query heads) and sliding-window attention with a
  configurable pattern such as "SSSL" of short and long windows; item 5: the
  flash-attention call takes a causal flag and a window.

Pins: closed forms (a window of one position returns each position's own
value; equal keys give the running mean over the window), special cases that
reduce to the unrestricted model (a window at least as long as the sequence,
an all-"L" pattern), a library routine (PyTorch scaled_dot_product_attention
with GQA and an explicit band mask), an independent scalar brute-force model
with groups and windows, decode == prefill with windows, GQA == MHA with each
group's K/V replicated, and planted mistakes that these pins catch.
"""
import cmath
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import nc_inputs
import oracle.gpt_oracle as go


def shape(**kw):
    base = dict(n_layer=2, d_model=32, n_head=4, n_kv_head=2, head_dim=8, d_mlp=64, vocab=48, dtype="f32")
    base.update(kw)
    return nc_inputs.ModelShape("t", **{k: base[k] for k in (
        "n_layer", "d_model", "n_head", "n_kv_head", "head_dim", "d_mlp", "vocab")},
        dtype=base["dtype"], window=base.get("window", 0), window_pattern=base.get("window_pattern", ""))


# ------------------------------------------------------------ attention ---- #

def check_window_attention(mod=go):
    rng = np.random.default_rng(5)
    T, nh, nkv, hd = 11, 4, 2, 8
    G = nh // nkv
    q = rng.standard_normal((T, nh, hd))
    k = rng.standard_normal((T, nkv, hd))
    v = rng.standard_normal((T, nkv, hd))
    pos = np.arange(T)
    full = mod.causal_attention(q, k, v, pos, pos)
    # a window as long as the sequence changes nothing
    if not np.array_equal(mod.causal_attention(q, k, v, pos, pos, T), full):
        return False
    # a window of one position: every query sees only its own key
    o1 = mod.causal_attention(q, k, v, pos, pos, 1)
    want1 = np.stack([v[:, h // G, :] for h in range(nh)], axis=1)
    if not np.allclose(o1, want1, rtol=1e-15, atol=0):
        return False
    # equal keys: the running mean of v over the last W positions
    W = 3
    ke = np.broadcast_to(rng.standard_normal((1, nkv, hd)), (T, nkv, hd)).copy()
    oe = mod.causal_attention(q, ke, v, pos, pos, W)
    for t in range(T):
        lo = max(0, t - W + 1)
        mean = v[lo:t + 1].mean(axis=0)                       # [nkv, hd]
        if not np.allclose(oe[t], mean[[h // G for h in range(nh)]], rtol=1e-12, atol=1e-14):
            return False
    # library routine: SDPA with GQA and an explicit band mask
    band = torch.from_numpy((pos[None, :] <= pos[:, None]) & (pos[None, :] > pos[:, None] - W))
    ref = F.scaled_dot_product_attention(torch.from_numpy(q).permute(1, 0, 2)[None],
                                         torch.from_numpy(k).permute(1, 0, 2)[None],
                                         torch.from_numpy(v).permute(1, 0, 2)[None],
                                         attn_mask=band, enable_gqa=True)
    ow = mod.causal_attention(q, k, v, pos, pos, W)
    if not np.allclose(ow, ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13):
        return False
    # GQA without a window against the same routine
    ref = F.scaled_dot_product_attention(torch.from_numpy(q).permute(1, 0, 2)[None],
                                         torch.from_numpy(k).permute(1, 0, 2)[None],
                                         torch.from_numpy(v).permute(1, 0, 2)[None],
                                         is_causal=True, enable_gqa=True)
    if not np.allclose(full, ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13):
        return False
    # decode form: the query at the last position over the cached keys
    return np.allclose(mod.causal_attention(q[-1:], k, v, [T - 1], pos, W), ow[-1:], rtol=1e-14, atol=1e-15)


def test_window_and_group_attention_pins():
    assert check_window_attention()


def test_layer_window_follows_the_pattern():
    s = shape(n_layer=8, window=5, window_pattern="SSSL")
    assert [go.layer_window(s, l) for l in range(8)] == [5, 5, 5, 0, 5, 5, 5, 0]
    assert [go.layer_window(shape(n_layer=3, window=5), l) for l in range(3)] == [0, 0, 0]
    assert [go.layer_window(shape(n_layer=3, window_pattern="S"), l) for l in range(3)] == [0, 0, 0]


# ----------------------------------------------------------- whole model --- #

def brute_force_logits(flat, s, tokens):
    """Scalar loops: K/V head of query head h = h // (n_head / n_kv), RoPE as a
    complex rotation, an explicit mask with the window of each layer."""
    d, hd, nh, nkv, V, Fm = s.d_model, s.head_dim, s.n_head, s.n_kv_head, s.vocab, s.d_mlp
    G = nh // nkv
    w = [float(t) for t in flat]
    idx = [0]

    def mat(r, c):
        m = [w[idx[0] + i * c: idx[0] + (i + 1) * c] for i in range(r)]
        idx[0] += r * c
        return m

    def mv(m, x):
        return [sum(a * b for a, b in zip(row, x)) for row in m]

    def nrm(x):
        ms = sum(t * t for t in x) / len(x)
        return [t / math.sqrt(ms + s.rms_eps) for t in x]

    def rot(x, p):
        h = hd // 2
        out = [0.0] * hd
        for j in range(h):
            z = complex(x[j], x[j + h]) * cmath.exp(1j * p * s.rope_base ** (-2.0 * j / hd))
            out[j], out[j + h] = z.real, z.imag
        return out

    E = mat(V, d)
    layers = [(mat((nh + 2 * nkv) * hd, d), mat(d, nh * hd), mat(Fm, d), mat(d, Fm)) for _ in range(s.n_layer)]
    Wu = mat(V, d)
    T = len(tokens)
    xs = [nrm(E[t]) for t in tokens]
    for li, (Wqkv, Wo, Wfc, Wproj) in enumerate(layers):
        short = bool(s.window_pattern) and s.window > 0 and s.window_pattern[li % len(s.window_pattern)] == "S"
        qs, ks, vs = [], [], []
        for p in range(T):
            r = mv(Wqkv, nrm(xs[p]))
            qs.append([nrm(rot(r[h * hd:(h + 1) * hd], p)) for h in range(nh)])
            ks.append([nrm(rot(r[(nh + g) * hd:(nh + g + 1) * hd], p)) for g in range(nkv)])
            vs.append([r[(nh + nkv + g) * hd:(nh + nkv + g + 1) * hd] for g in range(nkv)])
        for p in range(T):
            att = []
            for h in range(nh):
                g = h // G
                seen = [j for j in range(T) if j <= p and (not short or j > p - s.window)]
                sc = {j: sum(a * b for a, b in zip(qs[p][h], ks[j][g])) / math.sqrt(hd) for j in seen}
                mx = max(sc.values())
                e = {j: math.exp(c - mx) for j, c in sc.items()}
                tot = sum(e.values())
                att += [sum(e[j] / tot * vs[j][g][i] for j in seen) for i in range(hd)]
            xs[p] = [a + b for a, b in zip(xs[p], mv(Wo, att))]
        for p in range(T):
            u = [max(t, 0.0) ** 2 for t in mv(Wfc, nrm(xs[p]))]
            xs[p] = [a + b for a, b in zip(xs[p], mv(Wproj, u))]
    return np.array([[s.softcap * math.tanh(z / s.softcap) for z in mv(Wu, nrm(x))] for x in xs])


@pytest.mark.parametrize("kw", [dict(n_kv_head=2), dict(n_kv_head=2, window=3, window_pattern="SL"),
                                dict(n_kv_head=1, window=2, window_pattern="LS"),
                                dict(n_kv_head=4, window=4, window_pattern="S")])
def test_brute_force_groups_and_windows(kw):
    s = shape(**kw)
    flat = nc_inputs.gen_weights(s, 150, std=0.3)
    tok = nc_inputs.gen_tokens(s.vocab, (1, 8), 151)
    got = go.OracleModel(flat, s).prefill(tok)[0]
    np.testing.assert_allclose(got, brute_force_logits(flat, s, tok[0]), rtol=0, atol=1e-12)


def check_windowed_model(mod=go):
    """Windows at least as long as the sequence, or an all-"L" pattern, give
    the unrestricted model; decode == prefill with short windows; an "S"
    layer with a short window changes the logits."""
    s = shape()
    flat = nc_inputs.gen_weights(s, 152, std=0.3)
    tok = nc_inputs.gen_tokens(s.vocab, (2, 12), 153)
    base = mod.OracleModel(flat, s).prefill(tok)
    if not np.array_equal(mod.OracleModel(flat, s.with_(window=12, window_pattern="S")).prefill(tok), base):
        return False
    if not np.array_equal(mod.OracleModel(flat, s.with_(window=3, window_pattern="L")).prefill(tok), base):
        return False
    sw = s.with_(window=4, window_pattern="SL")
    full = mod.OracleModel(flat, sw).prefill(tok)
    if np.allclose(full, base, atol=1e-6):
        return False
    o = mod.OracleModel(flat, sw)
    o.prefill(tok[:, :5])
    steps = [o.decode(tok[:, t]) for t in range(5, 12)]
    return np.allclose(np.stack(steps, axis=1), full[:, 5:], rtol=0, atol=1e-12)


def test_windowed_model_special_cases_and_decode():
    assert check_windowed_model()


def test_chunked_prefill_with_windows_and_groups_equals_whole_prefill():
    """A prompt prefilled in chunks (the second and third starting inside a
    window) gives the whole prefill's logits, with short "S" layers and
    grouped K/V heads: the chunk's queries see the window over keys cached by
    earlier chunks."""
    s = shape(n_kv_head=2, window=4, window_pattern="SL")
    flat = nc_inputs.gen_weights(s, 156, std=0.3)
    tok = nc_inputs.gen_tokens(s.vocab, (2, 13), 157)
    whole = go.OracleModel(flat, s).prefill(tok)
    o = go.OracleModel(flat, s)
    parts = [o.prefill(tok[:, :5]), o.extend(tok[:, 5:7]), o.extend(tok[:, 7:])]
    np.testing.assert_allclose(np.concatenate(parts, axis=1), whole, rtol=0, atol=1e-12)


def test_gqa_equals_mha_with_each_group_replicated():
    s = shape(n_kv_head=2)
    flat = nc_inputs.gen_weights(s, 154, std=0.3).astype(np.float64)
    tok = nc_inputs.gen_tokens(s.vocab, (1, 9), 155)
    gqa = go.OracleModel(flat, s).prefill(tok)
    E, layers, Wu = go.unpack_weights(flat, s)
    hd, nh, nkv = s.head_dim, s.n_head, s.n_kv_head
    G = nh // nkv
    parts = [E.ravel()]
    for L in layers:
        W = L["Wqkv"]
        q = W[:nh * hd]
        k = [W[(nh + g) * hd:(nh + g + 1) * hd] for g in range(nkv)]
        v = [W[(nh + nkv + g) * hd:(nh + nkv + g + 1) * hd] for g in range(nkv)]
        parts += [np.concatenate([q] + [k[h // G] for h in range(nh)] + [v[h // G] for h in range(nh)]).ravel(),
                  L["Wo"].ravel(), L["Wfc"].ravel(), L["Wproj"].ravel()]
    parts.append(Wu.ravel())
    mha = go.OracleModel(np.concatenate(parts), s.with_(n_kv_head=nh)).prefill(tok)
    np.testing.assert_allclose(gqa, mha, rtol=0, atol=1e-13)


# --------------------------------------------------- planted mistakes ------ #

_attn = go.causal_attention
_layer_window = go.layer_window


def _window_off_by_one(q, k, v, q_pos, k_pos, window=0):
    return _attn(q, k, v, q_pos, k_pos, window + 1 if window > 0 else 0)


def _groups_interleaved(q, k, v, q_pos, k_pos, window=0):
    nh, nkv = q.shape[1], k.shape[1]
    order = [h % nkv for h in range(nh)]                      # h % n_kv instead of h // G
    out = np.empty_like(q)
    for h in range(nh):
        out[:, h:h + 1] = _attn(q[:, h:h + 1], k[:, order[h]:order[h] + 1], v[:, order[h]:order[h] + 1],
                                q_pos, k_pos, window)
    return out


MUTANTS = {
    "window_off_by_one": ("causal_attention", _window_off_by_one),
    "groups_interleaved": ("causal_attention", _groups_interleaved),
    "pattern_inverted": ("layer_window", lambda s, li: (s.window if _layer_window(s, li) == 0 else 0)
                         if s.window_pattern and s.window > 0 else 0),
}


def _caught(monkeypatch, name, fn):
    monkeypatch.setattr(go, name, fn)
    for pin in (check_window_attention, check_windowed_model):
        try:
            if not pin(go):
                return True
        except Exception:
            return True
    return False


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(monkeypatch, mutant):
    name, fn = MUTANTS[mutant]
    assert _caught(monkeypatch, name, fn), f"no pin caught {mutant}"
