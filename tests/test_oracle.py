"""Pins for the float64 oracle (CPU only).

The oracle is checked against things other than itself:
  * golden fixtures derived by hand in closed form (tests/golden);
  * central finite differences of O in float64 (tO is a derivative);
  * torch.func.jvp of a naive torch float64 attention (an independent
    autodiff routine, the cross-check the JVP tests of "Flash Attention v2
    with JVP" use);
  * invariants and special cases: rows of P sum to 1, sum exp(S - LSE) = 1,
    one key gives O = V and tO = tV, Q = 0 gives a uniform average, zero
    tangents give tO = 0 exactly, tO is linear in the tangents, tV = V with
    tQ = tK = 0 gives tO = O, masked / future / out-of-sequence entries do
    not influence any output, jagged equals the dense oracle per sequence.
The last test plants mistakes in the oracle and checks that each one trips
at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attn_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def _num(x):
    if isinstance(x, list):
        return [_num(e) for e in x]
    if isinstance(x, str):
        return {"ln4": math.log(4.0), "ln3": math.log(3.0), "1+ln2": 1.0 + math.log(2.0),
                "2/3": 2.0 / 3.0, "-inf": -math.inf}[x]
    return float(x)


def _rand_case(rng, B=1, H=2, M=5, N=7, Dqk=4, Dv=3, bias=False, mask=False, scale=0.7):
    c = dict(
        q=rng.standard_normal((B, H, M, Dqk)), k=rng.standard_normal((B, H, N, Dqk)),
        v=rng.standard_normal((B, H, N, Dv)), tq=rng.standard_normal((B, H, M, Dqk)),
        tk=rng.standard_normal((B, H, N, Dqk)), tv=rng.standard_normal((B, H, N, Dv)),
        sm_scale=scale, bias=None, mask=None)
    if bias:
        c["bias"] = rng.standard_normal((B, H, M, N))
    if mask:
        m = rng.random((B, 1, 1, N)) < 0.7
        m[..., 0] = True  # keep every row non-empty
        c["mask"] = m
    return c


def _run(c, causal):
    return oracle.attention_fwd_jvp(c["q"], c["k"], c["v"], c["tq"], c["tk"], c["tv"],
                                    causal=causal, sm_scale=c["sm_scale"],
                                    bias=c["bias"], mask=c["mask"])


def _fwd_only(c, causal, q, k, v):
    return oracle.attention_fwd(q, k, v, causal=causal, sm_scale=c["sm_scale"],
                                bias=c["bias"], mask=c["mask"])


# ------------------------------------------------------------- pin checks
def pin_golden():
    for fn in sorted(os.listdir(GOLDEN)):
        if not fn.endswith(".json"):
            continue
        g = json.load(open(os.path.join(GOLDEN, fn)))
        arr = {k: np.array(_num(g[k])) for k in ("q", "k", "v", "tq", "tk", "tv")}
        if g["layout"] == "dense":
            O, tO, L = oracle.attention_fwd_jvp(
                arr["q"], arr["k"], arr["v"], arr["tq"], arr["tk"], arr["tv"],
                causal=g["causal"], sm_scale=g["sm_scale"],
                bias=np.array(_num(g["bias"])) if "bias" in g else None,
                mask=np.array(g["mask"]) if "mask" in g else None)
        else:
            O, tO, L = oracle.attention_fwd_jvp_jagged(
                arr["q"], arr["k"], arr["v"], arr["tq"], arr["tk"], arr["tv"],
                np.array(g["offsets"]), g["max_seq_len"], causal=g["causal"],
                sm_scale=g["sm_scale"])
        np.testing.assert_allclose(O, np.array(_num(g["O"])), rtol=0, atol=1e-13, err_msg=fn)
        np.testing.assert_allclose(tO, np.array(_num(g["tO"])), rtol=0, atol=1e-13, err_msg=fn)
        np.testing.assert_allclose(L, np.array(_num(g["LSE"])), rtol=0, atol=1e-13, err_msg=fn)


def pin_finite_difference(causal, bias, mask, M=5, N=7, seed=1):
    rng = np.random.default_rng(seed)
    c = _rand_case(rng, M=M, N=N, bias=bias, mask=mask)
    _, tO, _ = _run(c, causal)
    eps = 1e-6
    Op, _ = _fwd_only(c, causal, c["q"] + eps * c["tq"], c["k"] + eps * c["tk"], c["v"] + eps * c["tv"])
    Om, _ = _fwd_only(c, causal, c["q"] - eps * c["tq"], c["k"] - eps * c["tk"], c["v"] - eps * c["tv"])
    fd = (Op - Om) / (2 * eps)
    np.testing.assert_allclose(tO, fd, rtol=0, atol=1e-7 * max(1.0, np.abs(fd).max()))


def pin_finite_difference_jagged(seed=2):
    rng = np.random.default_rng(seed)
    H, D = 2, 4
    lens = [3, 1, 6, 2]
    off = np.concatenate([[0], np.cumsum(lens)])
    T = int(off[-1])
    q, k, v, tq, tk, tv = (rng.standard_normal((H, T, D)) for _ in range(6))
    _, tO, _ = oracle.attention_fwd_jvp_jagged(q, k, v, tq, tk, tv, off, 5, sm_scale=0.6)
    eps = 1e-6
    Op, _ = oracle.attention_fwd_jagged(q + eps * tq, k + eps * tk, v + eps * tv, off, 5, sm_scale=0.6)
    Om, _ = oracle.attention_fwd_jagged(q - eps * tq, k - eps * tk, v - eps * tv, off, 5, sm_scale=0.6)
    fd = (Op - Om) / (2 * eps)
    np.testing.assert_allclose(tO, fd, rtol=0, atol=1e-7 * max(1.0, np.abs(fd).max()))


def _naive_torch(q, k, v, sm_scale, causal, bias, mask):
    s = torch.matmul(q, k.transpose(-1, -2)) * sm_scale
    if bias is not None:
        s = s + bias
    M, N = s.shape[-2], s.shape[-1]
    keep = torch.ones((M, N), dtype=torch.bool)
    if causal:
        keep = torch.tril(keep)
    if mask is not None:
        keep = keep & mask
    s = s.masked_fill(~keep, float("-inf"))
    return torch.matmul(torch.softmax(s, dim=-1), v)


def pin_torch_func_jvp(causal, bias, mask, M=6, N=6, seed=3):
    rng = np.random.default_rng(seed)
    c = _rand_case(rng, M=M, N=N, bias=bias, mask=mask)
    O, tO, _ = _run(c, causal)
    t = {k: torch.from_numpy(np.ascontiguousarray(c[k])) for k in ("q", "k", "v", "tq", "tk", "tv")}
    tb = None if c["bias"] is None else torch.from_numpy(c["bias"])
    tm = None if c["mask"] is None else torch.from_numpy(c["mask"])
    fn = lambda q, k, v: _naive_torch(q, k, v, c["sm_scale"], causal, tb, tm)
    ref_o, ref_to = torch.func.jvp(fn, (t["q"], t["k"], t["v"]), (t["tq"], t["tk"], t["tv"]))
    np.testing.assert_allclose(O, ref_o.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(tO, ref_to.numpy(), rtol=0, atol=1e-11)


def pin_softmax_and_lse(causal, seed=4):
    rng = np.random.default_rng(seed)
    q, k = rng.standard_normal((6, 4)), rng.standard_normal((6, 4))
    ok = attn_ref.valid_keys(6, 6, causal)
    s = attn_ref.scores(q, k, 0.9)
    p, lse = attn_ref.softmax_rows(s, ok)
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=0, atol=1e-15)
    assert np.all(p[~ok] == 0.0)
    e = np.where(ok, np.exp(s - lse[:, None]), 0.0)
    np.testing.assert_allclose(e.sum(1), 1.0, rtol=0, atol=1e-14)
    # LSE against the library routine
    ref = np.array([np.logaddexp.reduce(s[i][ok[i]]) for i in range(6)])
    np.testing.assert_allclose(lse, ref, rtol=0, atol=1e-13)


def pin_one_key():
    rng = np.random.default_rng(5)
    c = _rand_case(rng, M=3, N=1, bias=True)
    O, tO, L = _run(c, False)
    np.testing.assert_allclose(O, np.broadcast_to(c["v"], O.shape), rtol=0, atol=1e-15)
    np.testing.assert_allclose(tO, np.broadcast_to(c["tv"], tO.shape), rtol=0, atol=1e-14)
    ref_l = c["sm_scale"] * np.einsum("bhmd,bhnd->bhm", c["q"], c["k"]) + c["bias"][..., 0]
    np.testing.assert_allclose(L, ref_l, rtol=0, atol=1e-14)


def pin_zero_query():
    rng = np.random.default_rng(6)
    c = _rand_case(rng, M=4, N=5)
    c["q"] = np.zeros_like(c["q"])
    O, _, L = _run(c, False)
    np.testing.assert_allclose(O, np.broadcast_to(c["v"].mean(axis=2, keepdims=True), O.shape),
                               rtol=0, atol=1e-15)
    np.testing.assert_allclose(L, math.log(5.0), rtol=0, atol=1e-15)


def pin_tangent_special_cases():
    rng = np.random.default_rng(7)
    c = _rand_case(rng, M=5, N=6, bias=True, mask=True)
    z = dict(c, tq=np.zeros_like(c["tq"]), tk=np.zeros_like(c["tk"]), tv=np.zeros_like(c["tv"]))
    _, tO0, _ = _run(z, True)
    assert np.all(tO0 == 0.0)
    w = dict(c, tq=np.zeros_like(c["tq"]), tk=np.zeros_like(c["tk"]), tv=c["v"].copy())
    O, tOv, _ = _run(w, True)
    np.testing.assert_allclose(tOv, O, rtol=0, atol=1e-14)
    # linearity in (tQ, tK, tV)
    c2 = _rand_case(np.random.default_rng(8), M=5, N=6)
    a = -1.7
    mix = dict(c, tq=a * c["tq"] + c2["tq"], tk=a * c["tk"] + c2["tk"], tv=a * c["tv"] + c2["tv"])
    o2 = dict(c, tq=c2["tq"], tk=c2["tk"], tv=c2["tv"])
    _, t1, _ = _run(c, True)
    _, t2, _ = _run(o2, True)
    _, tm, _ = _run(mix, True)
    np.testing.assert_allclose(tm, a * t1 + t2, rtol=0, atol=1e-12)


def pin_masked_entries_have_no_influence():
    rng = np.random.default_rng(9)
    c = _rand_case(rng, M=6, N=6, bias=True, mask=True)
    O, tO, L = _run(c, True)
    keep = np.tril(np.ones((6, 6), bool))[None, None] & c["mask"]
    d = {k: c[k].copy() for k in ("k", "v", "tk", "tv")}
    dead_keys = ~c["mask"][0, 0, 0]
    for nm in d:
        d[nm][:, :, dead_keys] += 1e3 * rng.standard_normal(d[nm][:, :, dead_keys].shape)
    bias = c["bias"].copy()
    bias[~np.broadcast_to(keep, bias.shape)] += 1e3
    c2 = dict(c, bias=bias, **d)
    O2, tO2, L2 = _run(c2, True)
    assert np.array_equal(O, O2) and np.array_equal(tO, tO2) and np.array_equal(L, L2)
    # a future key (causal) of row 0 does not influence row 0
    c3 = dict(c, k=c["k"].copy(), v=c["v"].copy())
    c3["k"][:, :, 5] += 10.0
    c3["v"][:, :, 5] += 10.0
    O3, tO3, L3 = _run(c3, True)
    assert np.array_equal(O[:, :, :5], O3[:, :, :5]) and np.array_equal(tO[:, :, :5], tO3[:, :, :5])


def pin_jagged_equals_dense_per_sequence():
    rng = np.random.default_rng(10)
    H, Dqk, Dv = 2, 4, 3
    lens = [4, 9, 1, 7]
    msl = 8
    off = np.concatenate([[0], np.cumsum(lens)])
    T = int(off[-1])
    q, k, tq, tk = (rng.standard_normal((H, T, Dqk)) for _ in range(4))
    v, tv = (rng.standard_normal((H, T, Dv)) for _ in range(2))
    for causal in (False, True):
        O, tO, L = oracle.attention_fwd_jvp_jagged(q, k, v, tq, tk, tv, off, msl, causal, 0.8)
        for i, n in enumerate(lens):
            b0 = off[i]
            kept = min(n, msl)
            sl = slice(b0, b0 + kept)
            dO, dtO, dL = oracle.attention_fwd_jvp(
                q[None, :, sl], k[None, :, sl], v[None, :, sl], tq[None, :, sl], tk[None, :, sl],
                tv[None, :, sl], causal=causal, sm_scale=0.8)
            np.testing.assert_array_equal(O[:, sl], dO[0])
            np.testing.assert_array_equal(tO[:, sl], dtO[0])
            np.testing.assert_array_equal(L[:, sl], dL[0])
            tail = slice(b0 + kept, b0 + n)
            assert np.all(O[:, tail] == 0) and np.all(tO[:, tail] == 0)
            assert np.all(L[:, tail] == -np.inf)


def pin_rows_helper_matches_full():
    rng = np.random.default_rng(11)
    c = _rand_case(rng, M=9, N=9, bias=True, mask=True)
    O, tO, L = _run(c, True)
    rows = [0, 3, 8]
    o, to, l = oracle.attention_fwd_jvp_rows(c["q"], c["k"], c["v"], c["tq"], c["tk"], c["tv"],
                                              0, 1, rows, causal=True, sm_scale=c["sm_scale"],
                                              bias=c["bias"], mask=c["mask"])
    np.testing.assert_allclose(o, O[0, 1, rows], rtol=0, atol=1e-14)
    np.testing.assert_allclose(to, tO[0, 1, rows], rtol=0, atol=1e-14)
    np.testing.assert_allclose(l, L[0, 1, rows], rtol=0, atol=1e-14)


ALL_PINS = [
    ("golden", pin_golden),
    ("fd_dense", lambda: pin_finite_difference(False, False, False)),
    ("fd_causal_bias_mask", lambda: pin_finite_difference(True, True, True, M=6, N=6)),
    ("fd_cross", lambda: pin_finite_difference(False, True, False, M=3, N=8)),
    ("fd_jagged", pin_finite_difference_jagged),
    ("jvp_dense", lambda: pin_torch_func_jvp(False, False, False)),
    ("jvp_causal_bias_mask", lambda: pin_torch_func_jvp(True, True, True)),
    ("softmax_lse", lambda: (pin_softmax_and_lse(False), pin_softmax_and_lse(True))),
    ("one_key", pin_one_key),
    ("zero_query", pin_zero_query),
    ("tangent_special", pin_tangent_special_cases),
    ("masked_no_influence", pin_masked_entries_have_no_influence),
    ("jagged_vs_dense", pin_jagged_equals_dense_per_sequence),
    ("rows_helper", pin_rows_helper_matches_full),
]


@pytest.mark.parametrize("name,fn", ALL_PINS, ids=[n for n, _ in ALL_PINS])
def test_pin(name, fn):
    fn()


# ------------------------------------------------------ planted mistakes
def _m_tangent_drop_qtk(q, k, tq, tk, s):
    return s * (tq @ k.T)


def _m_tangent_no_scale(q, k, tq, tk, s):
    return tq @ k.T + q @ tk.T


def _m_tangent_wrong_operand(q, k, tq, tk, s):
    return s * (tq @ tk.T + q @ k.T)


def _m_tangent_sign(q, k, tq, tk, s):
    return s * (tq @ k.T - q @ tk.T)


def _m_out_drop_ptv(p, ts, v, tv, o):
    pts = p * ts
    return pts @ v - pts.sum(1)[:, None] * o


def _m_out_drop_rho(p, ts, v, tv, o):
    return p @ tv + (p * ts) @ v


def _m_out_rho_sign(p, ts, v, tv, o):
    pts = p * ts
    return p @ tv + pts @ v + pts.sum(1)[:, None] * o


def _m_out_tv_for_v(p, ts, v, tv, o):
    pts = p * ts
    return p @ tv + pts @ tv - pts.sum(1)[:, None] * o


def _m_scores_bias_scaled(q, k, s, bias=None):
    out = s * (q @ k.T)
    return out if bias is None else out + s * bias


def _m_scores_transposed(q, k, s, bias=None):
    out = s * (k @ q.T).T[::-1]
    return out if bias is None else out + bias


def _m_causal_off_by_one(m, n, causal, row_index=None, mask=None):
    rows = np.arange(m) if row_index is None else np.asarray(row_index)
    ok = np.ones((len(rows), n), dtype=bool)
    if causal:
        ok &= np.arange(n)[None, :] < rows[:, None] + 2
    if mask is not None:
        ok &= np.asarray(mask, dtype=bool)
    return ok


def _m_lse_base2(s, ok):
    p, lse = attn_ref.__dict__["_orig_softmax_rows"](s, ok)
    return p, lse / math.log(2.0)


def _m_seq_no_truncation(offsets, max_seq_len):
    off = np.asarray(offsets, dtype=np.int64)
    return [(int(off[i]), int(off[i + 1]), int(off[i + 1] - off[i])) for i in range(len(off) - 1)]


MUTANTS = [
    ("score_tangent", _m_tangent_drop_qtk),
    ("score_tangent", _m_tangent_no_scale),
    ("score_tangent", _m_tangent_wrong_operand),
    ("score_tangent", _m_tangent_sign),
    ("tangent_out", _m_out_drop_ptv),
    ("tangent_out", _m_out_drop_rho),
    ("tangent_out", _m_out_rho_sign),
    ("tangent_out", _m_out_tv_for_v),
    ("scores", _m_scores_bias_scaled),
    ("scores", _m_scores_transposed),
    ("valid_keys", _m_causal_off_by_one),
    ("softmax_rows", _m_lse_base2),
    ("_seq_bounds", _m_seq_no_truncation),
]


@pytest.mark.parametrize("target,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, target, mutant):
    monkeypatch.setitem(attn_ref.__dict__, "_orig_softmax_rows", attn_ref.softmax_rows)
    monkeypatch.setattr(attn_ref, target, mutant)
    tripped = []
    for name, fn in ALL_PINS:
        try:
            fn()
        except AssertionError:
            tripped.append(name)
        except (ValueError, IndexError):
            tripped.append(name + "(shape)")
    assert tripped, f"no pin caught the planted mistake {mutant.__name__}"
