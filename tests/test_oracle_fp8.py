"""Pins for the FP8 (e5m2) forward oracle (CPU only).

* the e5m2 rounding step against hand-derived values of the format (one
  sign, five exponent, two mantissa bits, bias 15): grid points stay, ties
  go to the even mantissa, the largest finite value and the subnormals;
* closed forms: weights {1, 1/2} (exact in e5m2) give the exact attention;
  a three-key case whose output changes if the weights are not rounded, if
  the row sum is taken after the rounding, or if the output is not rounded;
* LSE is the unrounded log-sum-exp; the output stays within the rounding
  bound of the float64 attention; causal and empty rows;
* planted mistakes, each tripping a pin.
"""
import math

import numpy as np
import pytest

from oracle import attn_fp8_ref as f8
from oracle import attn_ref


def test_round_e5m2_grid_and_ties():
    grid = [1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 0.5, 0.625, -1.75, 0.0]
    np.testing.assert_array_equal(f8.round_e5m2(grid), grid)
    # midpoints go to the even mantissa (00 or 10)
    np.testing.assert_array_equal(f8.round_e5m2([1.125, 1.375, 1.625, 1.875]), [1.0, 1.5, 1.5, 2.0])
    np.testing.assert_array_equal(f8.round_e5m2([1.1, 1.2, 3.2, -2.7]), [1.0, 1.25, 3.0, -2.5])
    # largest finite 1.75 * 2^15, smallest normal 2^-14, subnormals k * 2^-16
    np.testing.assert_array_equal(f8.round_e5m2([57344.0, 2.0 ** -14, 2.0 ** -16, 3 * 2.0 ** -16]),
                                  [57344.0, 2.0 ** -14, 2.0 ** -16, 3 * 2.0 ** -16])


def test_round_e5m2_error_bound():
    x = np.random.default_rng(0).uniform(-100, 100, 20000)
    x = x[np.abs(x) > 2.0 ** -14]
    r = f8.round_e5m2(x)
    assert np.all(np.abs(r - x) <= 2.0 ** -3 * np.abs(x) * (1 + 1e-12))


def test_two_keys_exact_weights():
    # S = [ln 2, 0] -> p = [1, 1/2] exactly; O = (v1 + v2 / 2) / 1.5
    q = np.array([[math.log(2.0)]])
    k = np.array([[1.0], [0.0]])
    v = np.array([[2.0, 1.0], [0.5, 1.0]])
    o, lse = f8.head_fwd_e5m2(q, k, v, 1.0)
    np.testing.assert_allclose(o, [[1.5, 1.0]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, [math.log(3.0)], rtol=1e-15)


def _three_keys(v):
    # weights 1, 0.6, 0.3 (S = [0, ln 0.6, ln 0.3]); e5m2 weights 1, 0.625,
    # 0.3125; the row sum 1.9 is taken before the rounding
    q = np.array([[1.0]])
    k = np.array([[0.0], [math.log(0.6)], [math.log(0.3)]])
    return f8.head_fwd_e5m2(q, k, np.asarray(v, dtype=np.float64), 1.0)


def test_three_keys_weight_rounding_and_sum():
    # 7 * 0.3125 / 1.9 = 1.151 -> 1.25 (unrounded weight: 7 * 0.3 / 1.9 = 1.105 -> 1.0)
    o, lse = _three_keys([[0.0], [0.0], [7.0]])
    assert o[0, 0] == 1.25
    np.testing.assert_allclose(lse, [math.log(1.9)], rtol=1e-14)
    # 2.15 / 1.9 = 1.132 -> 1.25 (sum of the rounded weights: 2.15 / 1.9375 = 1.110 -> 1.0)
    o, _ = _three_keys([[2.15], [0.0], [0.0]])
    assert o[0, 0] == 1.25
    # the output is rounded: 1.9 / 1.9 exact, 1.0 / 1.9 = 0.526 -> 0.5
    o, _ = _three_keys([[1.0], [0.0], [0.0]])
    assert o[0, 0] == 0.5


def _rand(shape, seed):
    return f8.round_e5m2(np.random.default_rng(seed).standard_normal(shape))


def test_lse_and_bound_against_float64():
    m, n, d = 9, 33, 16
    q, k, v = _rand((m, d), 1), _rand((n, d), 2), _rand((n, d), 3)
    for causal in (False, True):
        o, lse = f8.head_fwd_e5m2(q, k, v, 0.25, causal)
        o64, lse64 = attn_ref.head_fwd(q, k, v, 0.25, causal=causal)
        np.testing.assert_allclose(lse, lse64, rtol=0, atol=1e-12)
        # weights within 2^-3 relative, then the output rounding (2^-3)
        p, _ = attn_ref.softmax_rows(attn_ref.scores(q, k, 0.25),
                                     attn_ref.valid_keys(m, n, causal))
        bound = 2.0 ** -3 * (p @ np.abs(v)) + 2.0 ** -3 * np.abs(o64) * (1 + 2.0 ** -3) + 1e-12
        assert np.all(np.abs(o - o64) <= bound + 2.0 ** -3 * bound)


def test_bound_terms():
    # two keys, weights 2/3 and 1/3: B = sum w |v|, O = sum w v, by hand
    q = np.array([[math.log(2.0)]])
    k = np.array([[1.0], [0.0]])
    v = np.array([[2.0, -1.0], [-0.5, 3.0]])
    B, O = f8.e5m2_bound_terms(q, k, v, 1.0)
    np.testing.assert_allclose(B, [[2 * 2 / 3 + 0.5 / 3, 1 * 2 / 3 + 3 / 3]], rtol=1e-14)
    np.testing.assert_allclose(O, [[2 * 2 / 3 - 0.5 / 3, -2 / 3 + 1.0]], rtol=1e-14)
    # B bounds |O|; O equals the float64 attention
    qq, kk, vv = _rand((6, 8), 11), _rand((10, 8), 12), _rand((10, 8), 13)
    B, O = f8.e5m2_bound_terms(qq, kk, vv, 0.4, causal=True)
    assert np.all(B >= np.abs(O) - 1e-12)
    np.testing.assert_allclose(O, attn_ref.head_fwd(qq, kk, vv, 0.4, causal=True)[0], rtol=1e-12, atol=1e-14)


def test_empty_rows_and_no_keys():
    q, k, v = _rand((4, 8), 5), _rand((0, 8), 6), _rand((0, 8), 7)
    o, lse = f8.head_fwd_e5m2(q, k, v, 0.5)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_dense_wrapper_equals_heads():
    import torch
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1, 2, 5, 8, generator=g).to(torch.float8_e5m2)
    k = torch.randn(1, 2, 7, 8, generator=g).to(torch.float8_e5m2)
    v = torch.randn(1, 2, 7, 8, generator=g).to(torch.float8_e5m2)
    O, L = f8.attention_fwd_e5m2(q, k, v, sm_scale=0.3)
    for h in range(2):
        o, l = f8.head_fwd_e5m2(*(attn_ref.to_f64(t[0, h]) for t in (q, k, v)), 0.3)
        np.testing.assert_array_equal(O[0, h], o)
        np.testing.assert_array_equal(L[0, h], l)


# ------------------------------------------------------- planted mistakes
_HEAD = f8.head_fwd_e5m2


def _mutant_no_weight_rounding(q, k, v, sm_scale, causal=False):
    o64, lse = attn_ref.head_fwd(q, k, v, sm_scale, causal=causal)
    return f8.round_e5m2(o64), lse


def _mutant_rounded_sum(q, k, v, sm_scale, causal=False):
    ok = attn_ref.valid_keys(q.shape[0], k.shape[0], causal)
    s = np.where(ok, attn_ref.scores(q, k, sm_scale), -np.inf)
    mx = s.max(axis=1)
    pt = f8.round_e5m2(np.exp(s - mx[:, None]))
    return f8.round_e5m2((pt @ v) / pt.sum(axis=1)[:, None]), mx + np.log(np.exp(s - mx[:, None]).sum(1))


def _mutant_no_output_rounding(q, k, v, sm_scale, causal=False):
    ok = attn_ref.valid_keys(q.shape[0], k.shape[0], causal)
    s = np.where(ok, attn_ref.scores(q, k, sm_scale), -np.inf)
    mx = s.max(axis=1)
    p = np.exp(s - mx[:, None])
    return (f8.round_e5m2(p) @ v) / p.sum(axis=1)[:, None], mx + np.log(p.sum(1))


@pytest.mark.parametrize("mutant", [_mutant_no_weight_rounding, _mutant_rounded_sum,
                                    _mutant_no_output_rounding])
def test_planted_mistake_is_caught(monkeypatch, mutant):
    monkeypatch.setattr(f8, "head_fwd_e5m2", mutant)
    with pytest.raises(AssertionError):
        test_three_keys_weight_rounding_and_sum()
