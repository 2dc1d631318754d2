"""GPU parity at the edges of the method, through the C ABI, against the fp64
oracle on the same seeded inputs:

* logit softcap in saturation (the unembedding scaled by 100, so most
  pre-cap logits lie far beyond the cap of 15);
* causality: the logits of a prefix do not change when tokens are appended;
* decode for a batch wider than the decode GEMMs (160 rows), which runs the
  generic one-position forward pass instead of the skinny decode GEMMs.

Tolerances: bf16 max |dlogit| <= 3e-2 and mean <= 5e-3, as in every parity
test, except where a bound is derived below from the arithmetic.
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


def _scaled_unembedding(sh, seed, factor):
    """Packed weights with Wu scaled by `factor`, rounded again to bf16 so
    that the oracle and the GPU consume the same values."""
    flat = nc_inputs.gen_weights(sh, seed)
    n = sh.vocab * sh.d_model
    flat[-n:] = nc_inputs.round_to_bf16(flat[-n:] * np.float32(factor))
    return flat


def test_softcap_saturation_prefill_and_decode():
    """Wu x 100: pre-cap logits have a spread of about 55, so close to half of
    them lie beyond 2.65 c and saturate the cap c = 15.  Checked:
      * every GPU logit satisfies |logit| <= c;
      * where the oracle's logit is saturated (|logit| >= 0.99 c, i.e. the
        pre-cap value beyond 2.65 c) the bf16 tolerance holds: there the
        softcap's slope is below 0.02 and the error left is that of the tanh;
      * elsewhere the softcap is 1-Lipschitz, so the error is at most the
        pre-cap error, which scales with Wu: 100 x the bf16 bound 3e-2;
      * the sign of every logit with |oracle| > 0.5 agrees."""
    sh = small_bf16_shape(n_layer=2, vocab=4096)
    c = sh.softcap
    flat = _scaled_unembedding(sh, 81, 100.0)
    B, T, steps = 2, 96, 2
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 82)
    nxt = nc_inputs.gen_tokens(sh.vocab, (steps, B), 83)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + steps)
    outs = [(m.prefill(to_dev(prompt)).cpu().numpy(), o.prefill(prompt))]
    for t in range(steps):
        outs.append((m.decode_step(to_dev(nxt[t])).cpu().numpy(), o.decode(nxt[t])))
    m.sync()
    m.close()
    got = np.concatenate([g.reshape(-1) for g, _ in outs]).astype(np.float64)
    want = np.concatenate([w.reshape(-1) for _, w in outs])
    assert np.all(np.abs(got) <= c), float(np.abs(got).max())
    sat = np.abs(want) >= 0.99 * c
    assert sat.mean() > 0.4, f"only {sat.mean():.2f} of the logits saturate"
    check_close(got[sat], want[sat], "bf16", "softcap saturated logits (Wu x 100)")
    check_close(got[~sat], want[~sat], "bf16", "softcap unsaturated logits (Wu x 100, Lipschitz bound)",
                tol=(100 * 3e-2, 100 * 5e-3))
    big = np.abs(want) > 0.5
    assert np.all(np.sign(got[big]) == np.sign(want[big]))


def test_prefix_logits_unchanged_when_tokens_are_appended():
    """Causality on the GPU: prefill(T) and prefill(T + k) of the same prompt
    give the same logits at positions < T, within the bf16 tolerance (and
    each matches the oracle)."""
    sh = small_bf16_shape(n_layer=2, vocab=2048)
    flat = nc_inputs.gen_weights(sh, 85)
    B, T, k = 2, 200, 57
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T + k), 86)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + k)
    short = m.prefill(to_dev(prompt[:, :T])).cpu().numpy()
    m.kv_reset()
    long = m.prefill(to_dev(prompt)).cpu().numpy()
    m.sync()
    m.close()
    check_close(short, long[:, :T], "bf16", "causality: prefix of prefill(T+k) vs prefill(T)")
    check_close(long, oracle_for(flat, sh).prefill(prompt), "bf16", "causality: prefill(T+k) vs oracle")


def test_decode_wider_than_the_decode_gemms():
    """160 rows: wider than the 128-column decode GEMMs, so each decode step
    runs the generic forward pass over one position (CTA-pair prefill GEMMs at
    M = 160, the clustered decode attention, a per-step final norm that
    advances the device length).  Every row is checked at every step."""
    sh = small_bf16_shape(n_layer=2, vocab=2048)
    flat = nc_inputs.gen_weights(sh, 87)
    B, T, steps = 160, 33, 3
    prompt = nc_inputs.gen_tokens(sh.vocab, (B, T), 88)
    nxt = nc_inputs.gen_tokens(sh.vocab, (steps, B), 89)
    o = oracle_for(flat, sh)
    m = ncp.Model(sh, flat, max_batch=B, max_seq=T + steps)
    check_close(m.prefill(to_dev(prompt), last_only=True).cpu().numpy(),
                o.prefill(prompt, logit_positions=[T - 1])[:, 0], "bf16", "wide batch prefill (160 rows)")
    for t in range(steps):
        got = m.decode_step(to_dev(nxt[t])).cpu().numpy()
        check_close(got, o.decode(nxt[t]), "bf16", f"wide batch decode (160 rows) step {t}")
    m.sync()
    assert m.kv_length() == (T + steps, B)
    m.close()
