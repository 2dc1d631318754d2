"""ORACLE -- test infrastructure only (imported by tests/, smoke() and bench.py's
CPU baseline; never by the product path).

Plain fp64 numpy statement of the forward pass of the nanochat-style GPT, used
both as full-sequence prefill and as one-token decode over a KV cache.  Every
step is written out literally, in the pages' order, with no fusion and no
blocking; library matmuls are the only primitive used.

Pages cited (titles abbreviated):
  [yelogs]  yelogs.com story on the nanochat launch, section "technical details
            and official Q&A" (architecture answer).
  [geoz]    geoz.com.cn "NanoChat: Karpathy open-sources a low-cost LLM ...",
            section "development tricks".
  [apidog]  apidog.com/th "train your own ChatGPT for $50", section "how nanochat
            works": 1 GPT model, 3 precision handling, 5 flash attention,
            6 inference engine.
  [szyisi]  szyisi.cn "$100, 8000 lines, a hand-built ChatGPT clone", sections
            "pre-training" and inference engine paragraph.

Readings taken where the pages are silent or garbled (identical in the CUDA path):
  R1 RMSNorm eps = 1e-6, inside the square root; no learned scale [yelogs].
  R2 Norms: after the token embedding, before attention, before the MLP and
     before the unembedding (the last one is the Llama-like reading) [yelogs].
  R3 RoPE: theta_j = p * base**(-2j/hd), j < hd/2, half-split pairs (j, j+hd/2),
     y_j = x_j cos - x_{j+hd/2} sin, y_{j+hd/2} = x_j sin + x_{j+hd/2} cos;
     positions start at 0; table precomputed [geoz], [apidog 1].
  R4 QK-norm: parameter-free RMSNorm over hd of each query head and key head,
     applied after RoPE (the two commute exactly) [yelogs], [apidog 1].
  R5 attention scale 1/sqrt(hd) (the SDPA default) [apidog 5].
  R6 ReLU^2 = relu(x)**2 (the formula itself was lost in extraction) [yelogs].
  R7 softcap(z) = c * tanh(z / c), c = 15 [yelogs].
  R8 no biases anywhere [yelogs]; untied E and Wu [yelogs], [apidog 1].
  R9 weights enter as the bf16-rounded values for bf16 models, then fp64.
  R10 engine steps on either side of the pass [apidog 6], [szyisi inference
     engine]: a prompt may be prefilled in chunks (each chunk continues the
     cache); "batch generation clones the KV cache for parallel sampling" is
     read as copying one row's cache to every row of the batch.
  R12 grouped-query attention [apidog 1]: n_kv K/V heads, query head h reads
     K/V head h // (n_head / n_kv); one K/V head is multi-query attention.
  R13 sliding-window attention [apidog 1, 5] (a configurable pattern such as
     "SSSL" of short and long windows; the pages give no sizes): layer l uses
     the letter pattern[l % len(pattern)]; "S" limits a query at position p to
     the keys p - window + 1 .. p, "L" is the unrestricted causal window.  An
     empty pattern or window 0 leaves every layer unrestricted.
  R14 later-architecture extras [apidog 1, "performance tricks" and the
     value-embedding snippet; the autoresearch list names backout and smear]:
     value embeddings on alternate layers, read as the even layers 0, 2, ...:
     v += 3 sigmoid(h[:C] G_l^T) * VE_l[tok] per K/V head, h the block's
     normed input, C = ve_gate_channels (the pages give no width; 32);
     per-layer residual scaling before block i: x = resid_i x + x0_i x0, x0
     the residual that enters block 0; smear after the embedding norm:
     x_t += smear_lambda sigmoid(x_t[:24] . w) x_{t-1}, the previous token's
     embedding (nothing before the first position); backout after the last
     block: x -= backout_lambda x_mid, x_mid the residual after the first half
     of the blocks (block L // 2 - 1).  Each is off unless the shape enables it.
  R11 sampling (the pages name parallel sampling but not its rule; plainest
     reading): temperature 0 is greedy, the lowest index among equal maxima;
     otherwise the candidates are ordered by (logit descending, index
     ascending), the first top_k are kept (0 keeps all), p_i is proportional to
     exp((l_i - l_max) / temperature), and a uniform draw u in [0, 1) picks the
     first candidate whose cumulative probability exceeds u.  The cumulative
     weights C_j are summed in candidate order and the total is the last of
     them, so "cumulative probability exceeds u" is C_j > u * C_last.  The
     draws are inputs.
"""
from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------- #
# shapes and the packed weight layout (PyTorch Linear [out, in], apidog 3)
# --------------------------------------------------------------------------- #


def block_param_count(d_model, n_head, n_kv_head, head_dim, d_mlp):
    """Weights in one block: Wqkv, Wo, Wfc, Wproj (no biases, no norm gains)."""
    q = n_head * head_dim
    kv = n_kv_head * head_dim
    return (q + 2 * kv) * d_model + d_model * q + d_mlp * d_model + d_model * d_mlp


def total_param_count(n_layer, d_model, n_head, n_kv_head, head_dim, d_mlp, vocab):
    """Untied embedding and unembedding plus the blocks [yelogs]."""
    return vocab * d_model + n_layer * block_param_count(
        d_model, n_head, n_kv_head, head_dim, d_mlp) + vocab * d_model


def unpack_weights(flat, shape):
    """Split the canonical packed vector into fp64 matrices.

    Order: E[V,d]; per layer Wqkv[(n_h+2 n_kv) hd, d], Wo[d, n_h hd],
    Wfc[F, d], Wproj[d, F]; then Wu[V, d].
    """
    s = shape
    d, hd, V, F = s.d_model, s.head_dim, s.vocab, s.d_mlp
    q, kv = s.n_head * hd, s.n_kv_head * hd
    flat = np.asarray(flat)
    off = 0

    def take(rows, cols):
        nonlocal off
        m = flat[off:off + rows * cols].astype(np.float64).reshape(rows, cols)
        off += rows * cols
        return m

    E = take(V, d)
    layers = []
    for _ in range(s.n_layer):
        layers.append(dict(Wqkv=take(q + 2 * kv, d), Wo=take(d, q),
                           Wfc=take(F, d), Wproj=take(d, F)))
    Wu = take(V, d)
    if off + extras_count(shape) != flat.size:
        raise ValueError(f"packed weights: consumed {off + extras_count(shape)} of {flat.size} values")
    return E, layers, Wu


def _ve_layers(s):
    """Layers with a value embedding (R14): the even ones."""
    return list(range(0, s.n_layer, 2)) if getattr(s, "value_embeds", False) else []


def extras_count(s):
    """Parameters of the enabled extras (R14), stored after Wu."""
    n = 0
    for _ in _ve_layers(s):
        n += s.vocab * s.n_kv_head * s.head_dim + s.n_kv_head * s.ve_gate_channels
    if getattr(s, "resid_lambdas", False):
        n += 2 * s.n_layer
    if getattr(s, "smear", False):
        n += s.smear_channels + 1
    if getattr(s, "backout", False):
        n += 1
    return n


def unpack_extras(flat, s):
    """The extras' parameters after Wu (R14), in order: the value-embedding
    tables of the even layers [V, n_kv * hd], their gates [n_kv, C]; residual
    and x0 lambdas [L] each; smear gate [24] and lambda; backout lambda."""
    flat = np.asarray(flat)
    off = flat.size - extras_count(s)

    def take(n):
        nonlocal off
        a = flat[off:off + n].astype(np.float64)
        off += n
        return a

    ex = {"ve": {}, "ve_gate": {}}
    for l in _ve_layers(s):
        ex["ve"][l] = take(s.vocab * s.n_kv_head * s.head_dim).reshape(s.vocab, s.n_kv_head, s.head_dim)
    for l in _ve_layers(s):
        ex["ve_gate"][l] = take(s.n_kv_head * s.ve_gate_channels).reshape(s.n_kv_head, s.ve_gate_channels)
    if getattr(s, "resid_lambdas", False):
        ex["resid"], ex["x0"] = take(s.n_layer), take(s.n_layer)
    if getattr(s, "smear", False):
        ex["smear_gate"], ex["smear_lambda"] = take(s.smear_channels), take(1)[0]
    if getattr(s, "backout", False):
        ex["backout_lambda"] = take(1)[0]
    return ex


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


# --------------------------------------------------------------------------- #
# the operations, one by one
# --------------------------------------------------------------------------- #


def rms_norm(x, eps):
    """Parameter-free RMSNorm over the last axis (R1) [yelogs]."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps)


def rope_tables(positions, head_dim, base):
    """Precomputed rotary tables cos, sin of shape [len(positions), hd/2] (R3) [geoz]."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = base ** (-2.0 * j / head_dim)
    theta = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(theta), np.sin(theta)


def apply_rope(x, cos, sin):
    """Rotate pairs (j, j + hd/2) of the last axis by the per-position angles (R3).

    x: [T, heads, hd]; cos, sin: [T, hd/2].
    """
    half = x.shape[-1] // 2
    a, b = x[..., :half], x[..., half:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def causal_attention(q, k, v, q_pos, k_pos, window=0):
    """Causal multi-query / grouped-query attention (R5, R12) [yelogs], [apidog 1, 5].

    q: [Tq, n_head, hd]; k, v: [Tk, n_kv, hd]; query head h reads key/value
    head h // (n_head / n_kv) -- with one KV head every query head shares it.
    A query at position p sees the keys at positions <= p, and with a window
    W > 0 only those > p - W (R13).
    Returns [Tq, n_head, hd].
    """
    n_head, hd = q.shape[1], q.shape[2]
    n_kv = k.shape[1]
    group = n_head // n_kv
    kp, qp = np.asarray(k_pos)[None, :], np.asarray(q_pos)[:, None]
    allowed = kp <= qp                                                    # [Tq, Tk]
    if window > 0:
        allowed = allowed & (kp > qp - window)
    out = np.empty_like(q)
    for h in range(n_head):
        kh, vh = k[:, h // group, :], v[:, h // group, :]
        scores = (q[:, h, :] @ kh.T) / np.sqrt(hd)
        scores = np.where(allowed, scores, -np.inf)
        scores = scores - scores.max(axis=1, keepdims=True)
        p = np.exp(scores)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vh
    return out


def layer_window(shape, li):
    """Attention window of layer li (R13): the short window for an "S" of the
    pattern, 0 (unrestricted) otherwise."""
    pattern = getattr(shape, "window_pattern", "") or ""
    window = getattr(shape, "window", 0) or 0
    if not pattern or window <= 0:
        return 0
    return window if pattern[li % len(pattern)] == "S" else 0


def relu_squared(x):
    """ReLU^2 activation (R6) [yelogs], [geoz]."""
    return np.maximum(x, 0.0) ** 2


def softcap(z, cap):
    """Logit softcap cap * tanh(z / cap) (R7) [yelogs]."""
    return cap * np.tanh(z / cap)


# --------------------------------------------------------------------------- #
# the model
# --------------------------------------------------------------------------- #


class OracleModel:
    """fp64 forward pass with a per-layer KV cache (post-RoPE, post-QK-norm k; v).

    ``prefill(tokens[B, T])`` runs the full sequence from an empty cache and
    returns logits [B, T, V]; ``decode(tokens[B])`` appends one position per row
    and returns logits [B, V] [szyisi inference engine], [apidog 6].
    """

    def __init__(self, flat_weights, shape):
        self.s = shape
        self.E, self.layers, self.Wu = unpack_weights(flat_weights, shape)
        self.ex = unpack_extras(flat_weights, shape)
        self.reset()

    def reset(self):
        self.k_cache = [None] * self.s.n_layer     # each [B, len, n_kv, hd]
        self.v_cache = [None] * self.s.n_layer
        self.length = 0
        self.prev_tok = None                       # last token of each row (smear, R14)

    # one block over the new positions of every row
    def _block(self, li, x, positions, tokens=None):
        s, W = self.s, self.layers[li]
        B, T, _ = x.shape
        hd, nh, nkv = s.head_dim, s.n_head, s.n_kv_head
        cos, sin = rope_tables(positions, hd, s.rope_base)

        h = rms_norm(x, s.rms_eps)                                  # pre-attention norm
        qkv = h @ W["Wqkv"].T                                       # bias-free projection
        q = qkv[..., :nh * hd].reshape(B, T, nh, hd)
        k = qkv[..., nh * hd:(nh + nkv) * hd].reshape(B, T, nkv, hd)
        v = qkv[..., (nh + nkv) * hd:].reshape(B, T, nkv, hd)
        if li in self.ex["ve"]:                                     # value embedding (R14)
            C = s.ve_gate_channels
            gate = 3.0 * sigmoid(h[..., :C] @ self.ex["ve_gate"][li].T)   # [B, T, n_kv]
            v = v + gate[..., None] * self.ex["ve"][li][tokens]

        y = np.empty((B, T, nh, hd))
        new_k, new_v = [], []
        for b in range(B):
            qb = rms_norm(apply_rope(q[b], cos, sin), s.rms_eps)   # RoPE, then QK-norm
            kb = rms_norm(apply_rope(k[b], cos, sin), s.rms_eps)
            vb = v[b]
            if self.k_cache[li] is None:
                kc, vc = kb, vb
            else:
                kc = np.concatenate([self.k_cache[li][b], kb], axis=0)
                vc = np.concatenate([self.v_cache[li][b], vb], axis=0)
            new_k.append(kc)
            new_v.append(vc)
            k_pos = np.arange(kc.shape[0])
            y[b] = causal_attention(qb, kc, vc, positions, k_pos, layer_window(s, li))
        self.k_cache[li] = np.stack(new_k)
        self.v_cache[li] = np.stack(new_v)

        x = x + y.reshape(B, T, nh * hd) @ W["Wo"].T                # out-proj + residual
        h = rms_norm(x, s.rms_eps)                                  # pre-MLP norm
        x = x + relu_squared(h @ W["Wfc"].T) @ W["Wproj"].T          # ReLU^2 MLP + residual
        return x

    def _forward(self, tokens, logit_positions=None):
        s = self.s
        tokens = np.asarray(tokens)
        B, T = tokens.shape
        if np.any(tokens < 0) or np.any(tokens >= s.vocab):
            raise ValueError("token id out of range")
        positions = np.arange(self.length, self.length + T)
        x = rms_norm(self.E[tokens], s.rms_eps)                     # embedding, then norm
        ex = self.ex
        if "smear_gate" in ex:                                      # smear (R14)
            prev = np.zeros_like(x)
            prev[:, 1:] = x[:, :-1]
            if self.length > 0:
                prev[:, 0] = rms_norm(self.E[self.prev_tok], s.rms_eps)
            gate = ex["smear_lambda"] * sigmoid(x[..., :s.smear_channels] @ ex["smear_gate"])
            x = x + gate[..., None] * prev
        self.prev_tok = tokens[:, -1].copy()
        x0, x_mid = x, None
        for li in range(s.n_layer):
            if "resid" in ex:                                       # residual / x0 lambdas (R14)
                x = ex["resid"][li] * x + ex["x0"][li] * x0
            x = self._block(li, x, positions, tokens)
            if li == s.n_layer // 2 - 1:
                x_mid = x
        if "backout_lambda" in ex:                                  # backout (R14)
            x = x - ex["backout_lambda"] * (x_mid if x_mid is not None else 0.0)
        self.length += T
        if logit_positions is not None:
            x = x[:, logit_positions, :]
        h = rms_norm(x, s.rms_eps)                                  # final norm (R2)
        return softcap(h @ self.Wu.T, s.softcap)                    # unembed + softcap

    def prefill(self, tokens, logit_positions=None):
        """Logits [B, T, V] (or [B, len(logit_positions), V]) from an empty cache."""
        self.reset()
        return self._forward(tokens, logit_positions)

    def decode(self, tokens):
        """One new token per row at position ``self.length``; logits [B, V]."""
        if self.length == 0:
            raise RuntimeError("decode before prefill")
        tokens = np.asarray(tokens).reshape(-1, 1)
        return self._forward(tokens)[:, 0, :]

    def extend(self, tokens, logit_positions=None):
        """Chunked prefill (R10): T more positions per row after the cached
        ones, from ``self.length``; logits [B, T, V] (or the listed positions)."""
        if self.length == 0:
            raise RuntimeError("extend before prefill")
        return self._forward(tokens, logit_positions)

    def clone_row(self, src, n):
        """Batch generation (R10): the cache becomes n copies of row ``src``."""
        if self.length == 0:
            raise RuntimeError("clone before prefill")
        for li in range(self.s.n_layer):
            self.k_cache[li] = np.repeat(self.k_cache[li][src:src + 1], n, axis=0)
            self.v_cache[li] = np.repeat(self.v_cache[li][src:src + 1], n, axis=0)
        self.prev_tok = np.repeat(self.prev_tok[src:src + 1], n, axis=0)


# --------------------------------------------------------------------------- #
# sampling the next token (R11)
# --------------------------------------------------------------------------- #


def sample_tokens(logits, temperature, top_k, u):
    """Next token per row from logits [B, V] (R11).

    temperature == 0: argmax, the lowest index among equal maxima.  Otherwise
    the candidates are ordered by (logit descending, index ascending), the first
    top_k kept (top_k == 0 keeps all V), weighted by exp((l - l_max) / T),
    the weights summed in that order into cumulative weights C_j, and the
    first candidate with C_j > u[b] * C_last is taken.
    """
    logits = np.asarray(logits, dtype=np.float64)
    B, V = logits.shape
    u = np.asarray(u, dtype=np.float64).reshape(B)
    out = np.empty(B, dtype=np.int64)
    for b in range(B):
        row = logits[b]
        if temperature == 0:
            out[b] = int(np.flatnonzero(row == row.max())[0])
            continue
        order = sorted(range(V), key=lambda i: (-row[i], i))
        keep = order if top_k <= 0 else order[:top_k]
        w = [math.exp((row[i] - row[keep[0]]) / temperature) for i in keep]
        cums, c = [], 0.0                 # cumulative weights in candidate order
        for wi in w:
            c += wi
            cums.append(c)
        total = cums[-1]
        pick = keep[-1]
        for i, ci in zip(keep, cums):
            if ci > u[b] * total:
                pick = i
                break
        out[b] = pick
    return out
