"""Pins of the oracle's engine steps on either side of the forward pass:
chunked prefill, KV-cache row cloning for batch generation, and next-token
sampling (from the Engine description of apidog.com/th "train your own
ChatGPT", "how nanochat works" item 6: KV cache, prefill / decode, batch
generation by cloning the cache; the sampling rule is the plainest reading and
is stated in the oracle's header).

Sampling is pinned by closed forms: on a uniform grid of draws the inverse-CDF
picks each candidate a number of times within one of N * p_i, for hand-computed
p_i; ties and top_k = 1 reduce to the lowest-index argmax.  The model steps are
pinned by equivalences that hold exactly in exact arithmetic (fp64 here).
"""
import math

import numpy as np
import pytest

import nc_inputs
import oracle.gpt_oracle as go


def grid_counts(logits, temperature, top_k, n=600):
    u = (np.arange(n) + 0.5) / n
    toks = go.sample_tokens(np.repeat(np.asarray([logits], dtype=np.float64), n, axis=0), temperature, top_k, u)
    return np.bincount(toks, minlength=len(logits))


# ----------------------------------------------------------------- sampling --- #

def test_greedy_takes_lowest_index_among_equal_maxima():
    got = go.sample_tokens([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, -1.0, 5.0], [-2.0, -1.0, -1.5, -3.0]], 0, 0,
                           [0.9, 0.1, 0.5])
    assert got.tolist() == [1, 0, 1]


def test_top_k_one_is_greedy_for_any_draw():
    rng = np.random.default_rng(3)
    logits = np.round(rng.normal(size=(64, 50)), 1)           # rounding makes ties common
    want = go.sample_tokens(logits, 0, 0, np.zeros(64))
    for u in (0.0, 0.37, 0.999):
        assert np.array_equal(go.sample_tokens(logits, 0.7, 1, np.full(64, u)), want)
    assert np.array_equal(want, [int(np.flatnonzero(r == r.max())[0]) for r in logits])


def test_inverse_cdf_on_a_grid_matches_the_softmax():
    # logits (0, ln 2, ln 3) at temperature 1: p = (1, 2, 3) / 6
    c = grid_counts([0.0, math.log(2.0), math.log(3.0)], 1.0, 0)
    assert np.all(np.abs(c - np.array([100, 200, 300])) <= 1), c


def test_temperature_divides_the_logits():
    # logits (0, 2 ln 2) at temperature 2: weights (1/2, 1), p = (1/3, 2/3)
    c = grid_counts([0.0, 2.0 * math.log(2.0)], 2.0, 0)
    assert np.all(np.abs(c - np.array([200, 400])) <= 1), c
    # a very low temperature concentrates on the maximum
    c = grid_counts([0.3, 0.1, 0.2], 1e-3, 0)
    assert c.tolist() == [600, 0, 0]


def test_top_k_truncates_and_renormalises():
    # keep the two largest of (0, ln 2, ln 3): weights (3, 2) / 5; index 0 never drawn
    c = grid_counts([0.0, math.log(2.0), math.log(3.0)], 1.0, 2)
    assert c[0] == 0
    assert np.all(np.abs(c[1:] - np.array([240, 360])) <= 1), c


def test_candidate_order_is_logit_then_index():
    # equal logits: the cumulative walk visits indices in ascending order
    u = np.array([0.1, 0.4, 0.9])
    assert go.sample_tokens(np.zeros((3, 3)), 1.0, 0, u).tolist() == [0, 1, 2]
    # the largest logit comes first: a small draw takes it
    assert go.sample_tokens([[0.0, 4.0, 1.0]], 1.0, 0, [1e-9]).tolist() == [1]


# -------------------------------------------------------- engine model steps --- #

@pytest.fixture(scope="module")
def tiny():
    w = nc_inputs.WORKLOADS["tiny"]
    return w.shape, nc_inputs.gen_weights(w.shape, w.weight_seed)


def test_chunked_prefill_equals_one_prefill(tiny):
    shape, flat = tiny
    toks = nc_inputs.gen_tokens(shape.vocab, (2, 40), 11)
    whole = go.OracleModel(flat, shape).prefill(toks)
    m = go.OracleModel(flat, shape)
    first = m.prefill(toks[:, :17])
    mid = m.extend(toks[:, 17:30])
    last = m.extend(toks[:, 30:])
    np.testing.assert_allclose(np.concatenate([first, mid, last], axis=1), whole, rtol=0, atol=1e-10)
    assert m.length == 40
    # a decode after the chunks equals a decode after the one prefill
    nxt = nc_inputs.gen_tokens(shape.vocab, (2,), 12)
    ref = go.OracleModel(flat, shape)
    ref.prefill(toks)
    np.testing.assert_allclose(m.decode(nxt), ref.decode(nxt), rtol=0, atol=1e-10)


def test_cloned_row_decodes_like_a_repeated_prompt(tiny):
    shape, flat = tiny
    prompts = nc_inputs.gen_tokens(shape.vocab, (2, 24), 13)
    nxt = nc_inputs.gen_tokens(shape.vocab, (2, 4), 14)
    for src in (0, 1):
        m = go.OracleModel(flat, shape)
        m.prefill(prompts)
        m.clone_row(src, 4)
        ref = go.OracleModel(flat, shape)
        ref.prefill(np.repeat(prompts[src:src + 1], 4, axis=0))
        for t in range(2):
            np.testing.assert_allclose(m.decode(nxt[t]), ref.decode(nxt[t]), rtol=0, atol=1e-10)
    # the clone really copies row `src`: rows 0 and 1 differ, so cloning the
    # wrong one would not match
    a, b = go.OracleModel(flat, shape), go.OracleModel(flat, shape)
    a.prefill(prompts)
    b.prefill(prompts)
    a.clone_row(0, 4)
    b.clone_row(1, 4)
    assert np.max(np.abs(a.decode(nxt[0]) - b.decode(nxt[0]))) > 1e-3


def test_engine_steps_refuse_an_empty_cache(tiny):
    shape, flat = tiny
    m = go.OracleModel(flat, shape)
    with pytest.raises(RuntimeError):
        m.extend(np.zeros((1, 3), dtype=np.int64))
    with pytest.raises(RuntimeError):
        m.clone_row(0, 2)


# --------------------------------------------------------- planted mistakes --- #

def _sample_variant(logits, temperature, top_k, u, ascending=False, temp_mul=False, keep_last=False,
                    greedy_last=False):
    logits = np.asarray(logits, dtype=np.float64)
    B, V = logits.shape
    u = np.asarray(u, dtype=np.float64).reshape(B)
    out = np.empty(B, dtype=np.int64)
    for b in range(B):
        row = logits[b]
        if temperature == 0:
            idx = np.flatnonzero(row == row.max())
            out[b] = int(idx[-1] if greedy_last else idx[0])
            continue
        order = sorted(range(V), key=lambda i: ((row[i] if ascending else -row[i]), i))
        keep = order if top_k <= 0 else (order[-top_k:] if keep_last else order[:top_k])
        w = np.array([math.exp((row[i] - row[keep[0]]) * temperature if temp_mul
                               else (row[i] - row[keep[0]]) / temperature) for i in keep])
        cum, pick = 0.0, keep[-1]
        for i, wi in zip(keep, w):
            cum += wi
            if cum > u[b] * w.sum():
                pick = i
                break
        out[b] = pick
    return out


def _clone_always_row0(self, src, n):
    go_clone(self, 0, n)


def _extend_restarts_positions(self, tokens, logit_positions=None):
    keep = self.length
    self.length = 0                                          # positions restart at 0
    out = self._forward(tokens, logit_positions)
    self.length += keep
    return out


go_clone = go.OracleModel.clone_row
SAMPLE_MUTANTS = {
    "sample_ascending": dict(ascending=True),
    "sample_temperature_multiplied": dict(temp_mul=True),
    "top_k_keeps_smallest": dict(keep_last=True),
    "greedy_last_index": dict(greedy_last=True),
}
ENGINE_PINS = [test_greedy_takes_lowest_index_among_equal_maxima, test_top_k_one_is_greedy_for_any_draw,
               test_inverse_cdf_on_a_grid_matches_the_softmax, test_temperature_divides_the_logits,
               test_top_k_truncates_and_renormalises, test_candidate_order_is_logit_then_index]
MODEL_PINS = [test_chunked_prefill_equals_one_prefill, test_cloned_row_decodes_like_a_repeated_prompt]


def _some_pin_fails(pins, *args):
    for pin in pins:
        try:
            pin(*args)
        except (AssertionError, RuntimeError, ValueError):
            return True
    return False


@pytest.mark.parametrize("mutant", sorted(SAMPLE_MUTANTS))
def test_planted_sampling_mistake_is_caught(monkeypatch, mutant):
    kw = SAMPLE_MUTANTS[mutant]
    monkeypatch.setattr(go, "sample_tokens", lambda *a: _sample_variant(*a, **kw))
    assert _some_pin_fails(ENGINE_PINS), f"no pin caught {mutant}"


@pytest.mark.parametrize("attr,fn", [("clone_row", _clone_always_row0), ("extend", _extend_restarts_positions)])
def test_planted_engine_mistake_is_caught(monkeypatch, tiny, attr, fn):
    monkeypatch.setattr(go.OracleModel, attr, fn)
    assert _some_pin_fails(MODEL_PINS, tiny), f"no pin caught the planted {attr} mistake"
