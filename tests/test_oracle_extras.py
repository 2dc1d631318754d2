"""Pins of the oracle's later-architecture extras (reading R14), from
apidog.com/th "how nanochat works" item 1 (value embeddings mixed into v by
an input-dependent gate; per-layer residual and x0 lambdas; smear of the
previous token's embedding; backout of the mid-layer residual) and the same
page's list of autoresearch improvements (backout, smear).

Pins: the extras at their neutral values give the base model exactly; an
independent scalar brute force with every extra on; decode == prefill,
chunked prefill == prefill and a cloned row == its source (the smear reaches
back across calls); and planted mistakes that the pins catch.
"""
import math

import numpy as np
import pytest

import nc_inputs
import oracle.gpt_oracle as go


def shape(**kw):
    base = dict(name="x", n_layer=2, d_model=32, n_head=4, n_kv_head=2, head_dim=8, d_mlp=64, vocab=40,
                dtype="f32", value_embeds=True, resid_lambdas=True, smear=True, backout=True,
                ve_gate_channels=8, smear_channels=6)
    base.update(kw)
    return nc_inputs.ModelShape(**base)


def weights(s, seed, std=0.3):
    return nc_inputs.gen_weights(s, seed, std=std).astype(np.float64)


def neutral(flat, s):
    """The extras at neutral values: zero tables, residual lambdas 1, x0,
    smear and backout lambdas 0."""
    flat = flat.copy()
    off = flat.size - go.extras_count(s)
    for name, cnt in nc_inputs.extras_layout(s):
        flat[off:off + cnt] = 1.0 if name == "resid_lambdas" else 0.0
        off += cnt
    return flat


def test_neutral_extras_are_the_base_model():
    s = shape(n_layer=3)
    flat = weights(s, 200)
    tok = nc_inputs.gen_tokens(s.vocab, (2, 9), 201)
    base_s = s.with_(value_embeds=False, resid_lambdas=False, smear=False, backout=False)
    base = go.OracleModel(flat[:flat.size - go.extras_count(s)], base_s).prefill(tok)
    np.testing.assert_array_equal(go.OracleModel(neutral(flat, s), s).prefill(tok), base)
    assert not np.allclose(go.OracleModel(flat, s).prefill(tok), base, atol=1e-3)


def brute_force_logits(flat, s, tokens):
    """Scalar loops written from reading R14: smear of the previous token's
    normed embedding, x0 = the residual entering block 0, lambdas before
    each block, value embeddings on even layers gated by 3 sigmoid(h[:C] . g),
    backout of the residual after block L // 2 - 1."""
    d, hd, nh, nkv, V, Fm = s.d_model, s.head_dim, s.n_head, s.n_kv_head, s.vocab, s.d_mlp
    G, L, C, SC = nh // nkv, s.n_layer, s.ve_gate_channels, s.smear_channels
    w = [float(t) for t in flat]
    idx = [0]

    def take(n):
        a = w[idx[0]:idx[0] + n]
        idx[0] += n
        return a

    def mat(r, c):
        return [take(c) for _ in range(r)]

    def mv(m, x):
        return [sum(a * b for a, b in zip(row, x)) for row in m]

    def nrm(x):
        ms = sum(t * t for t in x) / len(x)
        return [t / math.sqrt(ms + s.rms_eps) for t in x]

    def rot(x, p):
        out = [0.0] * hd
        for j in range(hd // 2):
            th = p * s.rope_base ** (-2.0 * j / hd)
            out[j] = x[j] * math.cos(th) - x[j + hd // 2] * math.sin(th)
            out[j + hd // 2] = x[j] * math.sin(th) + x[j + hd // 2] * math.cos(th)
        return out

    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    E = mat(V, d)
    blocks = [(mat((nh + 2 * nkv) * hd, d), mat(d, nh * hd), mat(Fm, d), mat(d, Fm)) for _ in range(L)]
    Wu = mat(V, d)
    even = list(range(0, L, 2))
    ve = {l: mat(V, nkv * hd) for l in even}
    veg = {l: mat(nkv, C) for l in even}
    resid, x0l = take(L), take(L)
    sg, sl = take(SC), take(1)[0]
    bl = take(1)[0]
    T = len(tokens)
    emb = [nrm(E[t]) for t in tokens]
    xs = []
    for p in range(T):
        g = sl * sig(sum(a * b for a, b in zip(emb[p][:SC], sg)))
        prev = emb[p - 1] if p > 0 else [0.0] * d
        xs.append([a + g * b for a, b in zip(emb[p], prev)])
    x0 = [list(x) for x in xs]
    mid = None
    for li, (Wqkv, Wo, Wfc, Wproj) in enumerate(blocks):
        xs = [[resid[li] * a + x0l[li] * b for a, b in zip(xs[p], x0[p])] for p in range(T)]
        qs, ks, vs = [], [], []
        for p in range(T):
            h = nrm(xs[p])
            r = mv(Wqkv, h)
            qs.append([nrm(rot(r[i * hd:(i + 1) * hd], p)) for i in range(nh)])
            ks.append([nrm(rot(r[(nh + j) * hd:(nh + j + 1) * hd], p)) for j in range(nkv)])
            vv = [r[(nh + nkv + j) * hd:(nh + nkv + j + 1) * hd] for j in range(nkv)]
            if li in ve:
                for j in range(nkv):
                    gate = 3.0 * sig(sum(a * b for a, b in zip(h[:C], veg[li][j])))
                    vv[j] = [a + gate * b for a, b in zip(vv[j], ve[li][tokens[p]][j * hd:(j + 1) * hd])]
            vs.append(vv)
        new = []
        for p in range(T):
            att = []
            for i in range(nh):
                j = i // G
                sc = [sum(a * b for a, b in zip(qs[p][i], ks[t][j])) / math.sqrt(hd) for t in range(p + 1)]
                mx = max(sc)
                e = [math.exp(c - mx) for c in sc]
                tot = sum(e)
                att += [sum(e[t] / tot * vs[t][j][k] for t in range(p + 1)) for k in range(hd)]
            new.append([a + b for a, b in zip(xs[p], mv(Wo, att))])
        xs = new
        for p in range(T):
            u = [max(t, 0.0) ** 2 for t in mv(Wfc, nrm(xs[p]))]
            xs[p] = [a + b for a, b in zip(xs[p], mv(Wproj, u))]
        if li == L // 2 - 1:
            mid = [list(x) for x in xs]
    xs = [[a - bl * b for a, b in zip(xs[p], mid[p])] for p in range(T)]
    return np.array([[s.softcap * math.tanh(z / s.softcap) for z in mv(Wu, nrm(x))] for x in xs])


def check_brute_force(mod=go):
    s = shape(n_layer=3)
    flat = weights(s, 202)
    tok = nc_inputs.gen_tokens(s.vocab, (1, 7), 203)
    got = mod.OracleModel(flat, s).prefill(tok)[0]
    return np.allclose(got, brute_force_logits(flat, s, tok[0]), rtol=0, atol=1e-12)


def test_brute_force_with_every_extra():
    assert check_brute_force()


def check_decode_chunk_clone(mod=go):
    s = shape(n_layer=2)
    flat = weights(s, 204)
    tok = nc_inputs.gen_tokens(s.vocab, (2, 12), 205)
    full = mod.OracleModel(flat, s).prefill(tok)
    o = mod.OracleModel(flat, s)
    o.prefill(tok[:, :5])
    dec = np.stack([o.decode(tok[:, t]) for t in range(5, 8)], axis=1)
    if not np.allclose(dec, full[:, 5:8], rtol=0, atol=1e-12):
        return False
    if not np.allclose(o.extend(tok[:, 8:]), full[:, 8:], rtol=0, atol=1e-12):
        return False
    c = mod.OracleModel(flat, s)
    c.prefill(tok[1:, :6])
    c.clone_row(0, 2)
    return np.allclose(c.decode(tok[1, 6:7].repeat(2)), full[[1, 1], 6], rtol=0, atol=1e-12)


def test_decode_chunk_and_clone_with_extras():
    assert check_decode_chunk_clone()


_sigmoid = go.sigmoid
MUTANTS = {
    "gate_tanh": ("sigmoid", lambda z: 0.5 * (1.0 + np.tanh(z))),          # a different squashing
    "gate_not_scaled": ("sigmoid", lambda z: _sigmoid(z) / 3.0 * 2.0),
    "ve_odd_layers": ("_ve_layers", lambda s: list(range(1, s.n_layer, 2)) if s.value_embeds else []),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(monkeypatch, mutant):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(go, name, fn)
    try:
        ok = check_brute_force(go)
    except Exception:
        ok = False
    assert not ok, f"no pin caught {mutant}"
