"""ORACLE -- test infrastructure, not part of the product.

A plain, slow, fp64 CPU statement of the nanochat-style GPT forward pass.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA path; the only
module both sides use is ``nc_inputs`` (seeded input generators).
"""
from .gpt_oracle import (  # noqa: F401
    OracleModel, unpack_weights, rms_norm, rope_tables, apply_rope, causal_attention,
    relu_squared, softcap, block_param_count, total_param_count, sample_tokens, layer_window,
    unpack_extras, extras_count, sigmoid,
)
