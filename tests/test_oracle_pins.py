"""Pins for the fp64 oracle: each check ties it to something other than itself
(hand-computed values, closed forms, invariants, library routines, a
brute-force scalar implementation, the pages' printed figures).

The mutation tests at the end plant plausible mistakes in the oracle (on the
CPU) and assert that at least one pin catches each of them.
"""
import cmath
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import nc_inputs
import oracle.gpt_oracle as go

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_shape(**kw):
    base = dict(name="t", n_layer=2, d_model=32, n_head=4, n_kv_head=1, head_dim=8,
                d_mlp=128, vocab=64, dtype="f32")
    base.update(kw)
    return nc_inputs.ModelShape(**base)


def page_figures():
    out = {}
    with open(os.path.join(GOLDEN, "page_figures.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (t.strip() for t in line.split("="))
                out[k] = float(v)
    return out


# ---------------------------------------------------------------- RMSNorm ---- #

def check_rmsnorm(mod=go):
    rng = np.random.default_rng(0)
    eps = 1e-6
    for scale in (1.0, 1e-3, 30.0):          # 1e-3: ms ~ eps, where eps placement shows
        x = rng.standard_normal((7, 48)) * scale
        y = mod.rms_norm(x, eps)
        ms = np.mean(x * x, axis=-1)
        want = np.sqrt(ms / (ms + eps))      # closed form of rms(y)
        if not np.allclose(np.sqrt(np.mean(y * y, axis=-1)), want, rtol=1e-12, atol=0):
            return False
    # hand value: [3, 4] has mean square 12.5
    y = mod.rms_norm(np.array([3.0, 4.0]), 0.0)
    if not np.allclose(y, np.array([3.0, 4.0]) / math.sqrt(12.5), rtol=1e-15):
        return False
    # scale invariance for alpha > 0 (eps = 0)
    x = rng.standard_normal(16)
    return np.allclose(mod.rms_norm(5.0 * x, 0.0), mod.rms_norm(x, 0.0), rtol=1e-14)


def test_rmsnorm_pins():
    assert check_rmsnorm()


# ------------------------------------------------------------------- RoPE ---- #

def check_rope(mod=go):
    rng = np.random.default_rng(1)
    # hand values: hd = 2 has one pair with frequency 1 -> angle = position
    cos, sin = mod.rope_tables([1], 2, 10000.0)
    y = mod.apply_rope(np.array([[[1.0, 0.0]]]), cos, sin)
    if not np.allclose(y[0, 0], [math.cos(1.0), math.sin(1.0)], rtol=1e-15):
        return False
    # hd = 4, base 10000: pair j = 1 turns at 10000**(-1/2) = 0.01 rad per position
    cos, sin = mod.rope_tables([100], 4, 10000.0)
    y = mod.apply_rope(np.array([[[0.0, 1.0, 0.0, 0.0]]]), cos, sin)
    if not np.allclose(y[0, 0], [0.0, math.cos(1.0), 0.0, math.sin(1.0)], atol=1e-14):
        return False
    # identity at position 0
    x = rng.standard_normal((1, 3, 16))
    cos, sin = mod.rope_tables([0], 16, 10000.0)
    if not np.array_equal(mod.apply_rope(x, cos, sin), x):
        return False
    # per-pair norm preservation
    x = rng.standard_normal((5, 2, 16))
    cos, sin = mod.rope_tables(np.arange(5) * 37, 16, 10000.0)
    y = mod.apply_rope(x, cos, sin)
    pn = lambda t: t[..., :8] ** 2 + t[..., 8:] ** 2
    if not np.allclose(pn(x), pn(y), rtol=1e-13):
        return False
    # relative position: <rope(q, m), rope(k, n)> depends only on m - n
    q = rng.standard_normal((1, 1, 16))
    k = rng.standard_normal((1, 1, 16))

    def dot(m, n):
        cq, sq = mod.rope_tables([m], 16, 10000.0)
        ck, sk = mod.rope_tables([n], 16, 10000.0)
        return float(np.sum(mod.apply_rope(q, cq, sq) * mod.apply_rope(k, ck, sk)))
    if not math.isclose(dot(7, 3), dot(107, 103), rel_tol=1e-11):
        return False
    # complex-number statement: z_j = x_j + i x_{j+hd/2} is multiplied by e^{i theta_j}
    x = rng.standard_normal((1, 1, 16))
    cos, sin = mod.rope_tables([11], 16, 500.0)
    y = mod.apply_rope(x, cos, sin)
    for j in range(8):
        z = complex(x[0, 0, j], x[0, 0, j + 8]) * cmath.exp(1j * 11 * 500.0 ** (-2 * j / 16))
        if not (math.isclose(y[0, 0, j], z.real, abs_tol=1e-12)
                and math.isclose(y[0, 0, j + 8], z.imag, abs_tol=1e-12)):
            return False
    return True


def test_rope_pins():
    assert check_rope()


def test_qknorm_commutes_with_rope_and_bounds_scores():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((6, 3, 32)) * 3
    cos, sin = go.rope_tables(np.arange(6) + 5, 32, 10000.0)
    a = go.rms_norm(go.apply_rope(x, cos, sin), 1e-6)
    b = go.apply_rope(go.rms_norm(x, 1e-6), cos, sin)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)
    # after QK-norm, |q.k|/sqrt(hd) <= sqrt(hd) (Cauchy-Schwarz, each norm = sqrt(hd))
    q = go.rms_norm(rng.standard_normal((50, 32)) * 100, 1e-6)
    k = go.rms_norm(rng.standard_normal((50, 32)) * 100, 1e-6)
    assert np.max(np.abs(q @ k.T)) / math.sqrt(32) <= math.sqrt(32) * (1 + 1e-12)


# -------------------------------------------------------------- attention ---- #

def check_attention(mod=go):
    rng = np.random.default_rng(3)
    T, nh, hd = 9, 3, 8
    # one position: the output is v_0 exactly
    q = rng.standard_normal((1, nh, hd))
    k = rng.standard_normal((1, 1, hd))
    v = rng.standard_normal((1, 1, hd))
    o = mod.causal_attention(q, k, v, [0], [0])
    if not np.allclose(o, np.broadcast_to(v, o.shape), rtol=1e-15, atol=0):
        return False
    # equal keys: causal running mean of v (pins the inclusive causal bound)
    q = rng.standard_normal((T, nh, hd))
    k = np.broadcast_to(rng.standard_normal((1, 1, hd)), (T, 1, hd)).copy()
    v = rng.standard_normal((T, 1, hd))
    o = mod.causal_attention(q, k, v, np.arange(T), np.arange(T))
    want = np.cumsum(v[:, 0, :], axis=0) / np.arange(1, T + 1)[:, None]
    if not np.allclose(o, want[:, None, :], rtol=1e-12, atol=1e-14):
        return False
    # library routine: PyTorch scaled_dot_product_attention (fp64, causal, GQA)
    q = rng.standard_normal((T, nh, hd))
    k = rng.standard_normal((T, 1, hd))
    v = rng.standard_normal((T, 1, hd))
    o = mod.causal_attention(q, k, v, np.arange(T), np.arange(T))
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2)[None]
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True, enable_gqa=True)
    if not np.allclose(o, ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13):
        return False
    # MQA == MHA with the single K/V head replicated for every query head
    o_mha = mod.causal_attention(q, np.repeat(k, nh, axis=1), np.repeat(v, nh, axis=1),
                                 np.arange(T), np.arange(T))
    if not np.allclose(o, o_mha, rtol=1e-14, atol=1e-15):
        return False
    # decode form: the query at position p over cached keys 0..p
    o_last = mod.causal_attention(q[-1:], k, v, [T - 1], np.arange(T))
    return np.allclose(o_last, o[-1:], rtol=1e-14, atol=1e-15)


def test_attention_pins():
    assert check_attention()


# -------------------------------------------------------- MLP and softcap ---- #

def check_relu2(mod=go):
    x = np.array([-3.0, -0.5, 0.0, 0.5, 2.0, 7.0])
    return np.array_equal(mod.relu_squared(x), np.array([0.0, 0.0, 0.0, 0.25, 4.0, 49.0]))


def test_relu2_hand_values():
    assert check_relu2()


def test_softcap_properties():
    z = np.linspace(-1e4, 1e4, 20001)
    y = go.softcap(z, 15.0)
    assert np.all(np.abs(y) <= 15.0)
    assert np.all(np.abs(go.softcap(np.linspace(-200, 200, 1001), 15.0)) < 15.0)
    assert np.array_equal(go.softcap(-z, 15.0), -y)                       # odd
    assert np.all(np.diff(go.softcap(np.linspace(-50, 50, 1001), 15.0)) > 0)  # monotone
    small = np.linspace(-0.1, 0.1, 11)
    # c tanh(z/c) = z - z^3/(3c^2) + ... : near identity for |z| << c
    np.testing.assert_allclose(go.softcap(small, 15.0), small - small ** 3 / 675, atol=1e-9)


# ----------------------------------------------------- whole-model pins ---- #

def torch_library_logits(flat, shape, tokens):
    """The same model expressed with PyTorch library ops in fp64: F.embedding,
    F.rms_norm, F.linear, complex-number RoPE, F.scaled_dot_product_attention."""
    s = shape
    d, hd, nh, nkv, V, Fm = s.d_model, s.head_dim, s.n_head, s.n_kv_head, s.vocab, s.d_mlp
    w = torch.from_numpy(np.asarray(flat, dtype=np.float64))
    sizes = [V * d] + [((nh + 2 * nkv) * hd * d), d * nh * hd, Fm * d, d * Fm] * s.n_layer + [V * d]
    parts = list(torch.split(w, sizes))
    E = parts.pop(0).view(V, d)
    Wu = parts.pop().view(V, d)
    tok = torch.from_numpy(np.asarray(tokens)).long()
    B, T = tok.shape
    norm = lambda t: F.rms_norm(t, (t.shape[-1],), eps=s.rms_eps)
    pos = torch.arange(T, dtype=torch.float64)
    freq = s.rope_base ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    rot = torch.polar(torch.ones(T, hd // 2, dtype=torch.float64), pos[:, None] * freq[None, :])

    def rope(t):                      # t [B, heads, T, hd]; pairs (j, j + hd/2) as complex
        z = torch.complex(t[..., :hd // 2], t[..., hd // 2:]) * rot
        return torch.cat([z.real, z.imag], dim=-1)

    x = norm(F.embedding(tok, E))
    for li in range(s.n_layer):
        Wqkv, Wo, Wfc, Wproj = (parts[4 * li + i] for i in range(4))
        Wqkv = Wqkv.view(-1, d)
        qkv = F.linear(norm(x), Wqkv)
        q, k, v = torch.split(qkv, [nh * hd, nkv * hd, nkv * hd], dim=-1)
        q = norm(rope(q.view(B, T, nh, hd).transpose(1, 2)))
        k = norm(rope(k.view(B, T, nkv, hd).transpose(1, 2)))
        v = v.view(B, T, nkv, hd).transpose(1, 2)
        y = F.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
        x = x + F.linear(y.transpose(1, 2).reshape(B, T, nh * hd), Wo.view(d, nh * hd))
        x = x + F.linear(F.relu(F.linear(norm(x), Wfc.view(Fm, d))).square(), Wproj.view(d, Fm))
    z = F.linear(norm(x), Wu)
    return (s.softcap * torch.tanh(z / s.softcap)).numpy()


def check_model_vs_torch_library(mod=go):
    s = small_shape()
    flat = nc_inputs.gen_weights(s, 11, std=0.3)
    tok = nc_inputs.gen_tokens(s.vocab, (2, 7), 12)
    got = mod.OracleModel(flat, s).prefill(tok)
    return np.allclose(got, torch_library_logits(flat, s, tok), rtol=0, atol=1e-11)


def test_model_matches_torch_library_formulation():
    assert check_model_vs_torch_library()


def brute_force_logits(flat, s, tokens):
    """Scalar Python loops; multi-head attention with the KV head replicated,
    complex-number RoPE, an explicit dense causal mask."""
    d, hd, nh, V, Fm = s.d_model, s.head_dim, s.n_head, s.vocab, s.d_mlp
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
    layers = [(mat((nh + 2) * hd, d), mat(d, nh * hd), mat(Fm, d), mat(d, Fm))
              for _ in range(s.n_layer)]
    Wu = mat(V, d)
    T = len(tokens)
    xs = [nrm(E[t]) for t in tokens]
    for Wqkv, Wo, Wfc, Wproj in layers:
        qs, ks, vs = [], [], []
        for p in range(T):
            r = mv(Wqkv, nrm(xs[p]))
            qs.append([nrm(rot(r[h * hd:(h + 1) * hd], p)) for h in range(nh)])
            kh = nrm(rot(r[nh * hd:(nh + 1) * hd], p))
            vh = r[(nh + 1) * hd:(nh + 2) * hd]
            ks.append([kh] * nh)        # replicated per query head
            vs.append([vh] * nh)
        mask = [[1 if j <= i else 0 for j in range(T)] for i in range(T)]
        for p in range(T):
            att = []
            for h in range(nh):
                sc = [sum(a * b for a, b in zip(qs[p][h], ks[j][h])) / math.sqrt(hd)
                      if mask[p][j] else None for j in range(T)]
                mx = max(c for c in sc if c is not None)
                e = [math.exp(c - mx) if c is not None else 0.0 for c in sc]
                tot = sum(e)
                att += [sum(e[j] / tot * vs[j][h][i] for j in range(T)) for i in range(hd)]
            xs[p] = [a + b for a, b in zip(xs[p], mv(Wo, att))]
        for p in range(T):
            u = [max(t, 0.0) ** 2 for t in mv(Wfc, nrm(xs[p]))]
            xs[p] = [a + b for a, b in zip(xs[p], mv(Wproj, u))]
    return np.array([[s.softcap * math.tanh(z / s.softcap) for z in mv(Wu, nrm(x))] for x in xs])


def test_brute_force_tiny():
    s = small_shape(d_model=16, n_head=2, head_dim=8, d_mlp=64, vocab=32)
    flat = nc_inputs.gen_weights(s, 21, std=0.3)
    tok = nc_inputs.gen_tokens(s.vocab, (1, 6), 22)
    got = go.OracleModel(flat, s).prefill(tok)[0]
    np.testing.assert_allclose(got, brute_force_logits(flat, s, tok[0]), rtol=0, atol=1e-12)


def check_bigram_special_case(mod=go):
    """All block weights zero => logits = softcap(Wu rms(rms(E[tok])))."""
    s = small_shape()
    flat = nc_inputs.gen_weights(s, 31, std=0.5).astype(np.float64)
    d, V = s.d_model, s.vocab
    flat[V * d: flat.size - V * d] = 0.0
    tok = nc_inputs.gen_tokens(V, (2, 5), 32)
    got = mod.OracleModel(flat, s).prefill(tok)
    E = flat[:V * d].reshape(V, d)
    Wu = flat[flat.size - V * d:].reshape(V, d)
    e = E[tok]
    n1 = e / np.sqrt((e * e).mean(-1, keepdims=True) + s.rms_eps)
    n2 = n1 / np.sqrt((n1 * n1).mean(-1, keepdims=True) + s.rms_eps)
    z = n2 @ Wu.T
    return np.allclose(got, s.softcap * np.tanh(z / s.softcap), rtol=0, atol=1e-13)


def test_bigram_special_case():
    assert check_bigram_special_case()


def check_softcap_saturation(mod=go):
    s = small_shape()
    flat = nc_inputs.gen_weights(s, 41).astype(np.float64)
    flat[flat.size - s.vocab * s.d_model:] *= 100.0    # Wu x 100 so tanh saturates
    logits = mod.OracleModel(flat, s).prefill(nc_inputs.gen_tokens(s.vocab, (1, 4), 42))
    return np.max(np.abs(logits)) < s.softcap and np.max(np.abs(logits)) > 0.9 * s.softcap


def test_softcap_saturation_in_model():
    assert check_softcap_saturation()


def check_causality(mod=go):
    s = small_shape()
    flat = nc_inputs.gen_weights(s, 51, std=0.2)
    tok = nc_inputs.gen_tokens(s.vocab, (2, 10), 52)
    m = mod.OracleModel(flat, s)
    full = m.prefill(tok)
    short = m.prefill(tok[:, :6])
    # equal up to fp64 round-off: BLAS blocking depends on the matrix shape
    return np.allclose(full[:, :6], short, rtol=0, atol=1e-13)


def test_causality_prefix_unchanged():
    assert check_causality()


def check_decode_equals_prefill(mod=go):
    s = small_shape()
    flat = nc_inputs.gen_weights(s, 61, std=0.2)
    tok = nc_inputs.gen_tokens(s.vocab, (3, 9), 62)
    m = mod.OracleModel(flat, s)
    full = m.prefill(tok)
    m.prefill(tok[:, :5])
    steps = [m.decode(tok[:, t]) for t in range(5, 9)]
    if m.length != 9:
        return False
    return np.allclose(np.stack(steps, axis=1), full[:, 5:], rtol=0, atol=1e-12)


def test_decode_equals_prefill():
    assert check_decode_equals_prefill()


def test_batch_rows_independent():
    s = small_shape()
    flat = nc_inputs.gen_weights(s, 71, std=0.2)
    tok = nc_inputs.gen_tokens(s.vocab, (4, 6), 72)
    m = go.OracleModel(flat, s)
    full = m.prefill(tok)
    perm = [2, 0, 3, 1]
    np.testing.assert_array_equal(m.prefill(tok[perm]), full[perm])
    np.testing.assert_array_equal(m.prefill(tok[1:2]), full[1:2])


def test_mqa_equals_mha_with_replicated_kv_in_model():
    s = small_shape()
    flat = nc_inputs.gen_weights(s, 81, std=0.2).astype(np.float64)
    tok = nc_inputs.gen_tokens(s.vocab, (1, 7), 82)
    mqa = go.OracleModel(flat, s).prefill(tok)
    # rebuild the packed vector with n_kv = n_head: replicate the K and V rows
    E, layers, Wu = go.unpack_weights(flat, s)
    hd, nh, d = s.head_dim, s.n_head, s.d_model
    parts = [E.ravel()]
    for L in layers:
        W = L["Wqkv"]
        q, k, v = W[:nh * hd], W[nh * hd:(nh + 1) * hd], W[(nh + 1) * hd:]
        parts += [np.concatenate([q] + [k] * nh + [v] * nh).ravel(), L["Wo"].ravel(),
                  L["Wfc"].ravel(), L["Wproj"].ravel()]
    parts.append(Wu.ravel())
    mha = go.OracleModel(np.concatenate(parts), s.with_(n_kv_head=nh)).prefill(tok)
    np.testing.assert_allclose(mqa, mha, rtol=0, atol=1e-13)


def test_tiny_workload_logits_bounded_and_finite():
    w = nc_inputs.WORKLOADS["tiny"]
    flat = nc_inputs.gen_weights(w.shape, w.weight_seed)
    tok = nc_inputs.gen_tokens(w.shape.vocab, (w.batch, w.prompt_len), w.prompt_seed)
    m = go.OracleModel(flat, w.shape)
    logits = m.prefill(tok)
    assert logits.shape == (1, 64, 512)
    assert np.all(np.isfinite(logits)) and np.max(np.abs(logits)) < 15.0
    nxt = nc_inputs.gen_tokens(w.shape.vocab, (w.decode_steps, w.batch), w.decode_seed)
    for t in range(w.decode_steps):
        assert m.decode(nxt[t]).shape == (1, 512)
    assert m.length == 80 and m.k_cache[0].shape == (1, 80, 1, 64)


# ------------------------------------------------- bookkeeping vs pages ---- #

def test_parameter_count_matches_page_figure():
    g = page_figures()
    d, nh, hd = int(g["d20_channels"]), int(g["d20_heads"]), int(g["d20_head_dim"])
    mha = go.total_param_count(20, d, nh, nh, hd, 4 * d, int(g["vocab"]))
    assert mha == 560_988_160
    assert abs(mha - g["d20_params_approx"]) / g["d20_params_approx"] < 0.01
    # the multi-query model of this build has fewer parameters
    assert go.total_param_count(20, d, nh, 1, hd, 4 * d, 65536) == 502_005_760
    for name, want in (("tiny", 491_520), ("d12", 173_801_472), ("d20", 502_005_760),
                       ("d24", 776_994_816)):
        sh = nc_inputs.SHAPES[name]
        got = go.total_param_count(sh.n_layer, sh.d_model, sh.n_head, sh.n_kv_head,
                                   sh.head_dim, sh.d_mlp, sh.vocab)
        assert got == want == nc_inputs.param_count(sh)
    # 6 N D with D = 20 N reproduces the page's ~4e19 training FLOPs
    assert g["gpus"] * g["rows_per_gpu"] * g["row_tokens"] == g["tokens_per_step"]
    assert abs(6 * mha * 20 * mha / g["train_flops_approx"] - 1) < 0.1


def test_unpack_rejects_wrong_length():
    s = small_shape()
    with pytest.raises(ValueError):
        go.unpack_weights(np.zeros(nc_inputs.param_count(s) + 1), s)


def test_bf16_rounding_of_inputs():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3], dtype=np.float32)
    r = nc_inputs.round_to_bf16(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties to even -> 1
    assert r[0] == 1.0 and r[1] == 1.0 and r[2] == np.float32(1.015625) and r[3] == -2.5
    assert np.all((r.view(np.uint32) & 0xFFFF) == 0)
    t = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(r, t)


# --------------------------------------------------- planted mistakes ------ #

def _mutant_rope_sign(x, cos, sin):
    h = x.shape[-1] // 2
    a, b = x[..., :h], x[..., h:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([a * c + b * s, -a * s + b * c], axis=-1)


def _mutant_rope_interleaved(x, cos, sin):
    a, b = x[..., 0::2], x[..., 1::2]
    c, s = cos[:, None, :], sin[:, None, :]
    out = np.empty_like(x)
    out[..., 0::2], out[..., 1::2] = a * c - b * s, a * s + b * c
    return out


def _mutant_attention_strict_mask(q, k, v, q_pos, k_pos):
    return go_causal(q, k, v, np.asarray(q_pos) - 1, k_pos)


def _mutant_attention_scale(q, k, v, q_pos, k_pos):
    return go_causal(q * math.sqrt(q.shape[-1]) ** -1, k, v, q_pos, k_pos)


go_causal = go.causal_attention
MUTANTS = {
    "rms_eps_outside": ("rms_norm", lambda x, eps: x / (np.sqrt(np.mean(x * x, -1, keepdims=True)) + eps)),
    "rms_no_mean": ("rms_norm", lambda x, eps: x / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps)),
    "rope_sign": ("apply_rope", _mutant_rope_sign),
    "rope_interleaved": ("apply_rope", _mutant_rope_interleaved),
    "rope_freq": ("rope_tables", lambda p, hd, base: go_rope_tables(p, hd, base * 2)),
    "attn_strict_mask": ("causal_attention", _mutant_attention_strict_mask),
    "attn_scale": ("causal_attention", _mutant_attention_scale),
    "relu_not_squared": ("relu_squared", lambda x: np.maximum(x, 0.0)),
    "gelu_like": ("relu_squared", lambda x: x * x),
    "no_softcap": ("softcap", lambda z, c: z),
}
go_rope_tables = go.rope_tables
PINS = [check_rmsnorm, check_rope, check_attention, check_relu2, check_model_vs_torch_library,
        check_bigram_special_case, check_softcap_saturation, check_causality,
        check_decode_equals_prefill]


def _caught(monkeypatch, name, fn):
    monkeypatch.setattr(go, name, fn)
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                if not pin(go):
                    return True
        except Exception:
            return True
    return False


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(monkeypatch, mutant):
    name, fn = MUTANTS[mutant]
    assert _caught(monkeypatch, name, fn), f"no pin caught the planted mistake {mutant}"
