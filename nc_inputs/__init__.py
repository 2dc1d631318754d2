"""Seeded synthetic inputs for the nanochat-style GPT forward pass.

This module is the only code shared between the fp64 oracle (``oracle/``) and
the CUDA path (``dense_gpt_transformer_fwd_b300``).  It holds the model shapes,
the workload table and the random-number recipes, and nothing of the model's
arithmetic: no norm, rotation, attention, activation or softcap lives here.

Sources for the shapes (pages on nanochat):
  * d20: 1280 channels, 10 heads of dim 128, 20 layers, vocab 2**16, rows of
    2048 tokens -- szyisi.cn article, "pre-training" section.
  * dense transformer, RoPE, QK norm, parameter-free RMSNorm, untied
    embedding/unembedding, ReLU^2, no biases, multi-query attention, logit
    softcap -- yelogs.com story, architecture Q&A.
  * d12/d24 widths follow the same depth rule: d_model = 64 * depth,
    heads = depth/2 of dim 128, MLP = 4 * d_model.

Canonical packed weight order (row-major ``[out, in]`` as a PyTorch Linear
stores it): ``E[V, d]``; then for each layer ``Wqkv[(n_head + 2 n_kv) * hd, d]``
(query heads, then key heads, then value heads), ``Wo[d, n_head * hd]``,
``Wfc[F, d]``, ``Wproj[d, F]``; then ``Wu[V, d]``.

Random recipe: every matrix entry is N(0, 0.02), drawn in that order from one
``numpy.random.default_rng(seed)`` stream as float32 standard normals times
0.02.  For bf16 workloads each value is then rounded to the nearest bf16
(ties to even), so both sides consume exactly the same, bf16-representable
numbers.  For fp8 workloads every projection matrix (Wqkv, Wo, Wfc, Wproj,
Wu) is rounded instead to a multiple of one power-of-two scale per matrix,
s = 2**ceil(log2(amax / 448)), by an FP8 E4M3 value (round to nearest even,
saturating at 448), and E to bf16.  Token ids are uniform over ``[0, V)`` from
``default_rng(seed)``.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

__all__ = [
    "ModelShape", "Workload", "SHAPES", "WORKLOADS", "param_count",
    "layer_param_count", "gen_weights", "gen_tokens", "round_to_bf16", "round_to_e4m3",
    "fp8_scale", "round_to_fp8_tensorwise", "weight_matrices", "extras_layout", "ve_layers",
]


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layer: int
    d_model: int
    n_head: int
    n_kv_head: int
    head_dim: int
    d_mlp: int
    vocab: int
    rope_base: float = 10000.0
    softcap: float = 15.0
    rms_eps: float = 1e-6
    dtype: str = "bf16"          # "bf16", "fp8" (FP8 E4M3 projection weights) or "f32"
    # sliding-window attention: layer l uses `window` (keys p - window + 1 .. p)
    # where window_pattern[l % len] is "S", the whole causal context for "L";
    # an empty pattern (the default) leaves every layer unrestricted
    window: int = 0
    window_pattern: str = ""
    # later-architecture extras (off by default): value embeddings on the even
    # layers with a gate over the first ve_gate_channels channels, per-layer
    # residual / x0 lambdas, smear over the first smear_channels channels,
    # backout of the mid-layer residual.  Their parameters follow Wu in the
    # packed vector (see extras_layout).
    value_embeds: bool = False
    resid_lambdas: bool = False
    smear: bool = False
    backout: bool = False
    ve_gate_channels: int = 32
    smear_channels: int = 24

    def with_(self, **kw) -> "ModelShape":
        return replace(self, **kw)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    batch: int
    prompt_len: int
    decode_steps: int
    weight_seed: int
    prompt_seed: int
    decode_seed: int | None

    @property
    def max_seq(self) -> int:
        return self.prompt_len + self.decode_steps


TINY = ModelShape("tiny", 2, 128, 2, 1, 64, 512, 512, dtype="f32")
D12 = ModelShape("d12", 12, 768, 6, 1, 128, 3072, 65536)
D20 = ModelShape("d20", 20, 1280, 10, 1, 128, 5120, 65536)
D24 = ModelShape("d24", 24, 1536, 12, 1, 128, 6144, 65536)
SHAPES = {s.name: s for s in (TINY, D12, D20, D24)}

# The five workloads: the tiny fp32 model (prefill + 16 decode steps), d12
# prefill 8 x 2048, d12 decode 32 x (512 + 256), d20 prefill 16 x 2048 and
# decode 64 x (1024 + 128), d24 prefill 8 x 2048 and decode 128 x (2048 + 128).
WORKLOADS = {w.name: w for w in (
    Workload("tiny", TINY, 1, 64, 16, 1000, 2000, 3000),
    Workload("d12_prefill", D12, 8, 2048, 0, 1012, 2012, None),
    Workload("d12_decode", D12, 32, 512, 256, 1012, 2112, 3012),
    Workload("d20_prefill", D20, 16, 2048, 0, 1020, 2020, None),
    Workload("d20_decode", D20, 64, 1024, 128, 1020, 2120, 3020),
    Workload("d24_prefill", D24, 8, 2048, 0, 1024, 2024, None),
    Workload("d24_decode", D24, 128, 2048, 128, 1024, 2124, 3024),
    # the d24 decode workload with FP8 projection weights (same seeds)
    Workload("d24_decode_fp8", D24.with_(name="d24_fp8", dtype="fp8"), 128, 2048, 128, 1024, 2124, 3024),
)}


def layer_param_count(s: ModelShape) -> int:
    """Weights of one block in the canonical order (QKV, O, FC, PROJ)."""
    hd = s.head_dim
    qkv = (s.n_head + 2 * s.n_kv_head) * hd * s.d_model
    o = s.d_model * s.n_head * hd
    mlp = 2 * s.d_mlp * s.d_model
    return qkv + o + mlp


def ve_layers(s: ModelShape) -> list[int]:
    """Layers with a value embedding: the even ones, 0, 2, 4, ..."""
    return list(range(0, s.n_layer, 2)) if s.value_embeds else []


def extras_layout(s: ModelShape):
    """(name, count) of the extras' parameters after Wu, in order: the value
    embedding tables VE_l [V][n_kv * hd] of every even layer, then their gate
    matrices G_l [n_kv][ve_gate_channels]; resid_lambdas [L], x0_lambdas [L];
    the smear gate [smear_channels] and smear_lambda [1]; backout_lambda [1]."""
    out = []
    for l in ve_layers(s):
        out.append((f"VE{l}", s.vocab * s.n_kv_head * s.head_dim))
    for l in ve_layers(s):
        out.append((f"VEgate{l}", s.n_kv_head * s.ve_gate_channels))
    if s.resid_lambdas:
        out += [("resid_lambdas", s.n_layer), ("x0_lambdas", s.n_layer)]
    if s.smear:
        out += [("smear_gate", s.smear_channels), ("smear_lambda", 1)]
    if s.backout:
        out.append(("backout_lambda", 1))
    return out


def param_count(s: ModelShape) -> int:
    """Length of the packed weight vector: E, the blocks, Wu, the extras."""
    return 2 * s.vocab * s.d_model + s.n_layer * layer_param_count(s) + sum(n for _, n in extras_layout(s))


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), returned as float32.

    Inputs are finite (normal draws), so no NaN/Inf handling is needed.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    r = ((u + bias) & np.uint32(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32)


E4M3_MAX = 448.0          # largest finite FP8 E4M3 value: 1.75 * 2**8
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_QUANTUM_MIN = 2.0 ** -9   # spacing of the subnormals


def round_to_e4m3(a: np.ndarray) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value (ties to even), saturating at
    +-448; returned as float32.  E4M3: 3 mantissa bits, exponent bias 7,
    normals from 2**-6, subnormals in steps of 2**-9."""
    x = np.asarray(a, dtype=np.float64)
    ax = np.abs(x)
    _, e2 = np.frexp(np.maximum(ax, E4M3_MIN_NORMAL))      # ax = f * 2**e2, f in [0.5, 1)
    quantum = np.ldexp(1.0, e2 - 1 - 3)                   # 3 mantissa bits below the leading one
    q = np.rint(ax / quantum) * quantum                  # np.rint rounds half to even
    q = np.minimum(q, E4M3_MAX)
    return (np.sign(x) * q).astype(np.float32)


def fp8_scale(a: np.ndarray) -> float:
    """Power-of-two tensor scale 2**ceil(log2(amax / 448)) (1 for an all-zero matrix)."""
    amax = float(np.max(np.abs(a))) if a.size else 0.0
    if amax == 0.0:
        return 1.0
    m, e = np.frexp(amax / E4M3_MAX)                      # amax / 448 = m * 2**e, m in [0.5, 1)
    return float(np.ldexp(1.0, int(e) - 1 if m == 0.5 else int(e)))


def round_to_fp8_tensorwise(a: np.ndarray) -> np.ndarray:
    """a rounded to s * e4m3(a / s) with the matrix's power-of-two scale s."""
    s = fp8_scale(a)
    return (round_to_e4m3(np.asarray(a, dtype=np.float64) / s).astype(np.float64) * s).astype(np.float32)


def weight_matrices(s: ModelShape):
    """(name, offset, rows, cols) of every matrix of the packed vector, in order."""
    d, hd, V, F = s.d_model, s.head_dim, s.vocab, s.d_mlp
    q, kv = s.n_head * hd, s.n_kv_head * hd
    out, off = [], 0
    for name, r, c in ([("E", V, d)] +
                       [(f"{n}{l}", r, c) for l in range(s.n_layer)
                        for n, r, c in (("Wqkv", q + 2 * kv, d), ("Wo", d, q), ("Wfc", F, d), ("Wproj", d, F))] +
                       [("Wu", V, d)]):
        out.append((name, off, r, c))
        off += r * c
    return out


def gen_weights(s: ModelShape, seed: int, std: float = 0.02) -> np.ndarray:
    """Packed float32 weight vector in canonical order, N(0, std^2) entries."""
    n = param_count(s)
    rng = np.random.default_rng(seed)
    w = rng.standard_normal(n, dtype=np.float32)
    w *= np.float32(std)
    # extras: the lambdas near their neutral values (residual 1, the others 0)
    # with a spread of 0.1, the tables and gates as drawn
    off = 2 * s.vocab * s.d_model + s.n_layer * layer_param_count(s)
    for name, cnt in extras_layout(s):
        seg = w[off:off + cnt]
        if name == "resid_lambdas":
            seg[:] = 1.0 + seg * np.float32(0.1 / std)
        elif name in ("x0_lambdas", "smear_lambda", "backout_lambda"):
            seg[:] = seg * np.float32(0.1 / std)
        off += cnt
    if s.dtype == "bf16":
        # chunked to bound the temporary memory on the largest models
        step = 1 << 26
        for i in range(0, n, step):
            w[i:i + step] = round_to_bf16(w[i:i + step])
    elif s.dtype == "fp8":
        for name, off, r, c in weight_matrices(s):
            seg = w[off:off + r * c]
            w[off:off + r * c] = round_to_bf16(seg) if name == "E" else round_to_fp8_tensorwise(seg)
    return w


def gen_tokens(vocab: int, shape: tuple[int, ...], seed: int) -> np.ndarray:
    """Uniform token ids over [0, vocab) as int32."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, vocab, size=shape, dtype=np.int32)
