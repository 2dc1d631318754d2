"""Pins of the FP8 input rounding (nc_inputs): the weights of an fp8 model are
rounded on the host to s * e4m3(w / s) with one power-of-two scale s per
matrix, and both the oracle and the GPU consume exactly these values.

Pins: the 256 E4M3 codes decoded bit by bit (independently of the function
under test), nearest-value rounding against that table by brute force, ties
to even, saturation, PyTorch's float8_e4m3fn conversion as a library routine,
and the scale rule.
"""
import numpy as np
import pytest
import torch

import nc_inputs


def e4m3_table():
    """Every finite E4M3 value, decoded from its bits: sign, 4 exponent bits
    (bias 7), 3 mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN."""
    vals = set()
    for code in range(256):
        sgn, exp, man = code >> 7, (code >> 3) & 0xF, code & 0x7
        if exp == 0xF and man == 0x7:
            continue
        v = (man / 8.0) * 2.0 ** -6 if exp == 0 else (1 + man / 8.0) * 2.0 ** (exp - 7)
        vals.add(-v if sgn else v)
    return np.array(sorted(vals))


def test_table_extremes():
    t = e4m3_table()
    assert t.max() == 448.0 and t.min() == -448.0
    assert np.min(t[t > 0]) == 2.0 ** -9
    assert len(t) == 253                   # 254 finite codes, +0 and -0 coincide


def test_rounding_is_nearest_with_ties_to_even():
    t = e4m3_table()
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(3000) * 40, rng.standard_normal(1000) * 1e-2,
                        (t[:-1] + t[1:]) / 2])                # every midpoint is a tie
    got = nc_inputs.round_to_e4m3(x).astype(np.float64)
    assert np.all(np.isin(got, t))
    dist = np.abs(t[None, :] - x[:, None])
    best = dist.min(axis=1)
    assert np.all(np.abs(got - x) == best)                     # a nearest value
    # at ties: the candidate with an even mantissa (its code is even)
    for xv, gv in zip(x[4000:], got[4000:]):
        lo, hi = t[t <= xv].max(), t[t >= xv].min()
        if lo != hi and xv - lo == hi - xv:
            a = abs(gv)
            code_m = int(round(a / 2.0 ** -9)) if a < 2.0 ** -6 else int(round((a / 2.0 ** np.floor(np.log2(a)) - 1) * 8))
            assert code_m % 2 == 0, (xv, gv)
    assert nc_inputs.round_to_e4m3(np.array([1.0625, 1.1875, 232.0]))[:].tolist() == [1.0, 1.25, 224.0]


def test_saturation_and_idempotence():
    t = e4m3_table()
    assert nc_inputs.round_to_e4m3(np.array([1000.0, -5000.0])).tolist() == [448.0, -448.0]
    np.testing.assert_array_equal(nc_inputs.round_to_e4m3(t), t.astype(np.float32))


def test_matches_torch_float8_conversion():
    rng = np.random.default_rng(8)
    x = np.clip(rng.standard_normal(100000) * 60, -448, 448)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(nc_inputs.round_to_e4m3(x).astype(np.float64), want)


@pytest.mark.parametrize("amax", [0.1, 448.0, 449.0, 3e-5, 1.0])
def test_scale_rule(amax):
    a = np.array([amax, -amax / 3])
    s = nc_inputs.fp8_scale(a)
    assert s > 0 and np.log2(s) == np.round(np.log2(s))       # a power of two
    assert amax / s <= 448.0 and amax / (s / 2) > 448.0      # the smallest such


def test_fp8_workload_weights():
    sh = nc_inputs.D12.with_(name="t", n_layer=1, d_model=256, n_head=2, d_mlp=512, vocab=512, dtype="fp8")
    w = nc_inputs.gen_weights(sh, 9).astype(np.float64)
    t = e4m3_table()
    for name, off, r, c in nc_inputs.weight_matrices(sh):
        m = w[off:off + r * c]
        if name == "E":
            np.testing.assert_array_equal(nc_inputs.round_to_bf16(m.astype(np.float32)), m.astype(np.float32))
            continue
        s = nc_inputs.fp8_scale(m)
        assert np.all(np.isin(m / s, t)), name
    assert sum(r * c for _, _, r, c in nc_inputs.weight_matrices(sh)) == nc_inputs.param_count(sh)
