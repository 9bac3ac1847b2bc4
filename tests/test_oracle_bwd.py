"""Pins for the float64 backward oracle (CPU only).

The backward oracle is checked against things other than itself:
  * torch.autograd through a naive float64 torch attention (an independent
    autodiff routine) for dense, causal, bias + mask and cross-attention
    heads;
  * central finite differences of the scalar loss sum(dO o O) along random
    directions in Q, K and V;
  * closed forms: one key gives dQ = dK = 0 and dV = the column sum of dO;
    Delta = rowsum(P o dP);
  * invariants: the softmax is unchanged when one vector is added to every
    key, so the rows of dK sum to zero; keys nobody attends get zero dK,
    dV; the jagged oracle equals the dense one per sequence.
The last test plants mistakes and checks that each one trips a pin.
"""
import numpy as np
import pytest
import torch

from oracle import attn_bwd_ref as bw
from oracle import attn_ref


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def _torch_grads(q, k, v, do, s, causal=False, bias=None, mask=None):
    """dQ, dK, dV of sum(dO * softmax(s Q K^T + bias) V) by torch.autograd
    (float64, masked keys at -inf)."""
    Q, K, V = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    S = s * Q @ K.T
    if bias is not None:
        S = S + torch.tensor(bias, dtype=torch.float64)
    ok = np.ones(S.shape, dtype=bool)
    if causal:
        ok &= np.arange(S.shape[1])[None, :] <= np.arange(S.shape[0])[:, None]
    if mask is not None:
        ok &= mask
    S = S.masked_fill(~torch.tensor(ok), float("-inf"))
    P = torch.softmax(S, dim=1)
    P = torch.nan_to_num(P, nan=0.0)  # fully masked rows
    O = P @ V
    (O * torch.tensor(do, dtype=torch.float64)).sum().backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


CASES = [
    # m, n, dqk, dv, causal, bias, mask
    (7, 7, 8, 8, False, False, False),
    (9, 9, 4, 6, True, False, False),
    (5, 11, 8, 4, False, True, True),
    (13, 3, 4, 8, False, False, False),
]


@pytest.mark.parametrize("m,n,dqk,dv,causal,use_bias,use_mask", CASES)
def test_matches_torch_autograd(m, n, dqk, dv, causal, use_bias, use_mask):
    q, k, v = _rand((m, dqk), 1), _rand((n, dqk), 2), _rand((n, dv), 3)
    do = _rand((m, dv), 4)
    bias = _rand((m, n), 5) if use_bias else None
    mask = (_rand((m, n), 6) > -0.5) if use_mask else None
    if mask is not None:
        mask[1, :] = False  # a fully masked row
    s = 0.37
    dq, dk, dv_, _ = bw.head_bwd(q, k, v, do, s, causal, bias, mask)
    tq, tk, tv = _torch_grads(q, k, v, do, s, causal, bias, mask)
    np.testing.assert_allclose(dq, tq, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv_, tv, rtol=1e-11, atol=1e-12)


def test_finite_differences():
    m, n, d = 6, 9, 5
    q, k, v, do = _rand((m, d), 11), _rand((n, d), 12), _rand((n, d), 13), _rand((m, d), 14)
    s = 0.5

    def loss(q_, k_, v_):
        o, _ = attn_ref.head_fwd(q_, k_, v_, s, causal=True)
        return float((o * do).sum())

    dq, dk, dv, _ = bw.head_bwd(q, k, v, do, s, causal=True)
    eps = 1e-6
    for which, g in ((0, dq), (1, dk), (2, dv)):
        u = _rand(g.shape, 20 + which)
        args_p = [q, k, v]
        args_m = [q, k, v]
        args_p[which] = args_p[which] + eps * u
        args_m[which] = args_m[which] - eps * u
        fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        an = float((g * u).sum())
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (which, fd, an)


def test_one_key_closed_form():
    m, d = 5, 4
    q, k, v, do = _rand((m, d), 31), _rand((1, d), 32), _rand((1, d), 33), _rand((m, d), 34)
    dq, dk, dv, delta = bw.head_bwd(q, k, v, do, 0.7)
    assert np.allclose(dq, 0.0, atol=1e-14) and np.allclose(dk, 0.0, atol=1e-14)
    np.testing.assert_allclose(dv[0], do.sum(axis=0), rtol=1e-14)
    np.testing.assert_allclose(delta, do @ v[0], rtol=1e-14)


def test_delta_is_rowsum_p_dp():
    m, n, d = 8, 10, 6
    q, k, v, do = _rand((m, d), 41), _rand((n, d), 42), _rand((n, d), 43), _rand((m, d), 44)
    p, _ = attn_ref.softmax_rows(attn_ref.scores(q, k, 0.3), np.ones((m, n), bool))
    _, _, _, delta = bw.head_bwd(q, k, v, do, 0.3)
    np.testing.assert_allclose(delta, (p * (do @ v.T)).sum(axis=1), rtol=1e-12)


def test_dk_rows_sum_to_zero():
    # adding one vector c to every key leaves the softmax unchanged
    m, n, d = 7, 12, 5
    q, k, v, do = _rand((m, d), 51), _rand((n, d), 52), _rand((n, d), 53), _rand((m, d), 54)
    _, dk, _, _ = bw.head_bwd(q, k, v, do, 0.9, causal=False)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)


def test_unattended_keys_get_zero_gradients():
    m, n, d = 6, 8, 4
    q, k, v, do = _rand((m, d), 61), _rand((n, d), 62), _rand((n, d), 63), _rand((m, d), 64)
    mask = np.ones((m, n), bool)
    mask[:, 5] = False
    _, dk, dv, _ = bw.head_bwd(q, k, v, do, 0.5, mask=mask)
    assert np.all(dk[5] == 0.0) and np.all(dv[5] == 0.0)


def test_jagged_equals_dense_per_sequence():
    H, d = 2, 4
    lens = [3, 0, 5, 2]
    off = np.concatenate([[0], np.cumsum(lens)])
    T = int(off[-1])
    q, k, v, do = (_rand((H, T, d), 70 + i) for i in range(4))
    dQ, dK, dV, Dl = bw.attention_bwd_jagged(q, k, v, do, off, max_seq_len=4, causal=True,
                                            sm_scale=0.6)
    for i, L in enumerate(lens):
        n = min(L, 4)
        b0 = off[i]
        for h in range(H):
            sl = slice(b0, b0 + n)
            tail = slice(b0 + n, off[i + 1])
            assert np.all(dQ[h, tail] == 0) and np.all(dK[h, tail] == 0)
            if n == 0:
                continue
            eq, ek, ev, ed = bw.head_bwd(q[h, sl], k[h, sl], v[h, sl], do[h, sl], 0.6, causal=True)
            np.testing.assert_allclose(dQ[h, sl], eq, rtol=1e-13)
            np.testing.assert_allclose(dK[h, sl], ek, rtol=1e-13)
            np.testing.assert_allclose(dV[h, sl], ev, rtol=1e-13)


# ------------------------------------------------------- planted mistakes
_HEAD_BWD = bw.head_bwd  # the real function (the mutants below call it)


def _mutant_no_delta(q, k, v, do, s, causal=False, bias=None, mask=None, row_index=None):
    m, n = q.shape[0], k.shape[0]
    ok = attn_ref.valid_keys(m, n, causal, row_index, mask)
    p, _ = attn_ref.softmax_rows(attn_ref.scores(q, k, s, bias), ok)
    ds = p * (do @ v.T)
    return s * ds @ k, s * ds.T @ q, p.T @ do, np.zeros(m)


def _mutant_dk_unscaled(q, k, v, do, s, causal=False, bias=None, mask=None, row_index=None):
    dq, dk, dv, dl = _HEAD_BWD(q, k, v, do, s, causal, bias, mask, row_index)
    return dq, dk / s, dv, dl


def _mutant_dv_transposed_p(q, k, v, do, s, causal=False, bias=None, mask=None, row_index=None):
    m, n = q.shape[0], k.shape[0]
    dq, dk, dv, dl = _HEAD_BWD(q, k, v, do, s, causal, bias, mask, row_index)
    ok = attn_ref.valid_keys(m, n, causal, row_index, mask)
    p, _ = attn_ref.softmax_rows(attn_ref.scores(q, k, s, bias), ok)
    if m == n:
        dv = p @ do
    else:
        dv = dv * 1.0001
    return dq, dk, dv, dl


def _mutant_dq_with_v(q, k, v, do, s, causal=False, bias=None, mask=None, row_index=None):
    dq, dk, dv, dl = _HEAD_BWD(q, k, v, do, s, causal, bias, mask, row_index)
    if k.shape[1] == v.shape[1]:
        m, n = q.shape[0], k.shape[0]
        ok = attn_ref.valid_keys(m, n, causal, row_index, mask)
        p, _ = attn_ref.softmax_rows(attn_ref.scores(q, k, s, bias), ok)
        ds = p * (do @ v.T - dl[:, None])
        dq = s * ds @ v
    return dq, dk, dv, dl


@pytest.mark.parametrize("mutant", [_mutant_no_delta, _mutant_dk_unscaled, _mutant_dv_transposed_p,
                                    _mutant_dq_with_v])
def test_planted_mistake_is_caught(monkeypatch, mutant):
    monkeypatch.setattr(bw, "head_bwd", mutant)
    caught = 0
    for fn in (test_matches_torch_autograd, test_finite_differences, test_dk_rows_sum_to_zero,
               test_one_key_closed_form):
        try:
            if fn is test_matches_torch_autograd:
                for case in CASES:
                    fn(*case)
            else:
                fn()
        except AssertionError:
            caught += 1
    assert caught >= 1, mutant.__name__
