"""Float64 CPU oracle for fused attention forward + JVP.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
the benchmark's CPU-baseline / reference legs may import this module.  It
shares no code with the CUDA path: it materialises every intermediate
(S, tS, P, O, LSE, tO) from the plain definition, in float64, one head at a
time, with no tiling, no online rescaling and no fusion.

What it computes, per (batch, head) or per (sequence, head):

  S   = s * Q K^T + bias                        scores
  V   = valid keys (causal j <= i, mask, in-sequence)
  S   = -inf off V
  tS  = s * (tQ K^T + Q tK^T), 0 off V          score tangent, no bias tangent
  P   = softmax_rows(S)                         masked keys get weight 0
  O   = P V
  LSE = log sum_j exp(S_ij)                     natural log of scaled scores
  tO  = P tV + (P o tS) V - rowsum(P o tS) o O
  empty row (no valid key): O = tO = 0, LSE = -inf

Sources (the pages; code, so each step's "equation" is a code step):
  * "Flash Attention v2 with JVP" (flm/utils/jvp.py): ``_attn_fwd_inner``
    (score tangent ``tS_ij = (tq k + q tk) * sm_scale``, masked tangent set
    to zero, ``H_ij = p * tS_ij``, running ``r_i``), ``_attn_fwd`` epilogue
    (``tO = (acc_A + acc_B - r * acc) / l`` with ``acc`` already divided by
    ``l``; LSE stored as a natural log; empty-row guard) and
    ``_attention.forward`` (default ``sm_scale = Dqk ** -0.5``; causal only
    when the query and key lengths agree).
  * "_06_fused_attention_blockptr_jvp.py" (Triton fused attention with JVP):
    ``_attn_fwd`` epilogue, ``tO = g_acc/l - (mu/l) * O + p_tv_acc/l`` -- the
    same closed form written with the tangent sum called ``mu``.
  * "flash_attention.py" (triton_flashattn): ``_attn_fwd_inner`` -- the
    additive bias is added after the ``sm_scale`` product and is not scaled;
    a boolean mask with True = attend.
  * "triton_multi_head_jagged_flash_attention.py" (FBGEMM): jagged layout
    ``[H, T, D]`` with ``offsets[B + 1]``; a sequence's length is
    ``min(offsets[b+1] - offsets[b], max_seq_len)``.

Readings where the pages disagree or are silent (each also stated in the
design notes): masked keys get exactly zero weight (-inf, not -1e6); the
row maximum is taken over valid keys only; a fully masked row yields
O = tO = 0 and LSE = -inf; jagged rows past ``max_seq_len`` inside their
sequence are written as empty rows; the jagged scores use ``sm_scale`` and
no ``1 / max_seq_len`` factor.
"""
from __future__ import annotations

import numpy as np

try:  # torch is only used to up-cast bf16 tensors exactly
    import torch
except Exception:  # pragma: no cover
    torch = None

NEG_INF = -np.inf


def to_f64(x):
    """Exact up-cast of a bf16/fp32/bool torch tensor or array to float64."""
    if x is None:
        return None
    if torch is not None and isinstance(x, torch.Tensor):
        if x.dtype == torch.bool:
            return x.numpy()
        return x.detach().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def default_scale(dqk: int) -> float:
    """``sm_scale = Dqk ** -0.5`` when none is given (jvp.py,
    ``_attention.forward``)."""
    return float(dqk) ** -0.5


# --------------------------------------------------------------------------
# one head
# --------------------------------------------------------------------------
def scores(q, k, sm_scale, bias=None):
    """S = sm_scale * Q K^T + bias (flash_attention.py, ``_attn_fwd_inner``:
    ``qk * qk_scale`` then ``qk += bias``; the bias is not scaled)."""
    s = sm_scale * (q @ k.T)
    if bias is not None:
        s = s + bias
    return s


def score_tangent(q, k, tq, tk, sm_scale):
    """tS = sm_scale * (tQ K^T + Q tK^T): the tangent of the scaled scores
    with respect to (Q, K); the bias has no tangent (jvp.py,
    ``_attn_fwd_inner``: ``tS_ij = dot(tq, k) + dot(q, tk)`` then
    ``tS_ij *= sm_scale``)."""
    return sm_scale * (tq @ k.T + q @ tk.T)


def valid_keys(m, n, causal, row_index=None, mask=None):
    """Boolean [m, n] set of attended keys.  Causal keeps key j <= query i
    (jvp.py, ``_attn_fwd_inner`` stage 2: ``offs_m >= start_n + offs_n``);
    ``mask`` True = attend (flash_attention.py, ``IS_BIAS_BOOL``)."""
    rows = np.arange(m) if row_index is None else np.asarray(row_index)
    ok = np.ones((len(rows), n), dtype=bool)
    if causal:
        ok &= np.arange(n)[None, :] <= rows[:, None]
    if mask is not None:
        ok &= np.asarray(mask, dtype=bool)
    return ok


def softmax_rows(s, ok):
    """Row softmax over the valid keys, with its log-sum-exp.

    P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i), m_i the maximum over
    valid keys; invalid keys get weight exactly 0.  LSE_i is the natural
    log of sum_j exp(S_ij) (jvp.py, ``_attn_fwd`` epilogue stores
    ``(m + log2 l) * ln 2``).  A row with no valid key returns P = 0 and
    LSE = -inf.
    """
    s = np.where(ok, s, NEG_INF)
    any_ok = ok.any(axis=1)
    m = np.where(any_ok, np.max(s, axis=1), 0.0)
    e = np.where(ok, np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)
    safe_l = np.where(any_ok, l, 1.0)
    p = e / safe_l[:, None]
    lse = np.where(any_ok, m + np.log(safe_l), NEG_INF)
    return p, lse


def tangent_out(p, ts, v, tv, o):
    """tO = P tV + (P o tS) V - rowsum(P o tS) o O.

    The tangent of softmax(S) V: dP = P o (tS - rowsum(P o tS)), so
    tO = dP V + P tV.  jvp.py, ``_attn_fwd`` epilogue:
    ``(acc_A + acc_B - r * acc) / l`` with ``acc_A = sum p tv``,
    ``acc_B = sum (p tS) v``, ``r = sum p tS`` and ``acc`` = O.
    """
    pts = p * ts
    rho = pts.sum(axis=1)
    return p @ tv + pts @ v - rho[:, None] * o


def head_fwd_jvp(q, k, v, tq, tk, tv, sm_scale, causal=False, bias=None,
                 mask=None, row_index=None):
    """Forward + JVP of one head, float64.  q/tq: [m, Dqk]; k/tk: [n, Dqk];
    v/tv: [n, Dv]; bias: [m, n] or None; mask: [m, n] bool or None;
    row_index: global query index of each q row (for the causal rule).

    Returns (O [m, Dv], tO [m, Dv], LSE [m]).
    tO = P tV + (P o tS) V - rowsum(P o tS) o O  (jvp.py, ``_attn_fwd``
    epilogue; the same form as ``t_y_out`` in the Triton JVP tutorial).
    """
    m, n = q.shape[0], k.shape[0]
    ok = valid_keys(m, n, causal, row_index, mask)
    s = scores(q, k, sm_scale, bias)
    ts = np.where(ok, score_tangent(q, k, tq, tk, sm_scale), 0.0)
    p, lse = softmax_rows(s, ok)
    o = p @ v
    to = tangent_out(p, ts, v, tv, o)
    empty = ~ok.any(axis=1)
    o[empty] = 0.0
    to[empty] = 0.0
    return o, to, lse


def head_fwd(q, k, v, sm_scale, causal=False, bias=None, mask=None, row_index=None):
    """Forward only (O, LSE) of one head; the same definition without the
    tangent."""
    m, n = q.shape[0], k.shape[0]
    ok = valid_keys(m, n, causal, row_index, mask)
    p, lse = softmax_rows(scores(q, k, sm_scale, bias), ok)
    o = p @ v
    o[~ok.any(axis=1)] = 0.0
    return o, lse


# --------------------------------------------------------------------------
# dense [B, H, M, D]
# --------------------------------------------------------------------------
def _bh(x, b, h, shape_mn):
    if x is None:
        return None
    x = np.broadcast_to(x, x.shape[:2] + shape_mn) if x.ndim == 4 else x
    bb = b if x.shape[0] > 1 else 0
    hh = h if x.shape[1] > 1 else 0
    return np.broadcast_to(x[bb, hh], shape_mn)


def attention_fwd_jvp(q, k, v, tq, tk, tv, causal=False, sm_scale=None,
                      bias=None, mask=None):
    """Dense forward + JVP.  q, tq: [B, H, M, Dqk]; k, tk: [B, H, N, Dqk];
    v, tv: [B, H, N, Dv]; bias: [B|1, H|1, M|1, N] float; mask: same with
    bool/uint8 (nonzero = attend).  Returns float64 (O, tO, LSE) with
    shapes [B, H, M, Dv], [B, H, M, Dv], [B, H, M]."""
    q, k, v, tq, tk, tv = (to_f64(x) for x in (q, k, v, tq, tk, tv))
    bias = to_f64(bias)
    mask = None if mask is None else (to_f64(mask) != 0)
    B, H, M, _ = q.shape
    N, Dv = v.shape[2], v.shape[3]
    if sm_scale is None:
        sm_scale = default_scale(q.shape[3])
    O = np.zeros((B, H, M, Dv))
    tO = np.zeros((B, H, M, Dv))
    L = np.zeros((B, H, M))
    for b in range(B):
        for h in range(H):
            O[b, h], tO[b, h], L[b, h] = head_fwd_jvp(
                q[b, h], k[b, h], v[b, h], tq[b, h], tk[b, h], tv[b, h], sm_scale,
                causal, _bh(bias, b, h, (M, N)), _bh(mask, b, h, (M, N)))
    return O, tO, L


def attention_fwd(q, k, v, causal=False, sm_scale=None, bias=None, mask=None):
    """Dense forward only: (O, LSE)."""
    q, k, v = (to_f64(x) for x in (q, k, v))
    bias = to_f64(bias)
    mask = None if mask is None else (to_f64(mask) != 0)
    B, H, M, _ = q.shape
    N, Dv = v.shape[2], v.shape[3]
    if sm_scale is None:
        sm_scale = default_scale(q.shape[3])
    O = np.zeros((B, H, M, Dv))
    L = np.zeros((B, H, M))
    for b in range(B):
        for h in range(H):
            O[b, h], L[b, h] = head_fwd(q[b, h], k[b, h], v[b, h], sm_scale, causal,
                                        _bh(bias, b, h, (M, N)), _bh(mask, b, h, (M, N)))
    return O, L


def attention_fwd_jvp_rows(q, k, v, tq, tk, tv, b, h, rows, causal=False,
                           sm_scale=None, bias=None, mask=None):
    """Forward + JVP for selected query rows of head (b, h) of a dense
    problem, every key considered: the sampled check used at full size."""
    rows = np.asarray(rows)
    qq = to_f64(q[b, h])[rows]
    tqq = to_f64(tq[b, h])[rows]
    kk, vv, tkk, tvv = (to_f64(x[b, h]) for x in (k, v, tk, tv))
    if sm_scale is None:
        sm_scale = default_scale(qq.shape[1])
    N = kk.shape[0]

    def rows_of(x, as_bool):
        if x is None:
            return None
        xb = x[b if x.shape[0] > 1 else 0, h if x.shape[1] > 1 else 0]
        xb = to_f64(xb)
        xb = xb[rows] if xb.shape[0] > 1 else xb
        xb = np.broadcast_to(xb, (len(rows), N))
        return xb != 0 if as_bool else xb

    return head_fwd_jvp(qq, kk, vv, tqq, tkk, tvv, sm_scale, causal,
                        rows_of(bias, False), rows_of(mask, True), row_index=rows)


# --------------------------------------------------------------------------
# jagged [H, T, D] with offsets[B + 1]
# --------------------------------------------------------------------------
def _seq_bounds(offsets, max_seq_len):
    """(begin, end, kept length) per sequence: the kept length is
    ``min(end - begin, max_seq_len)`` (FBGEMM jagged attention forward)."""
    off = np.asarray(offsets, dtype=np.int64)
    out = []
    for i in range(len(off) - 1):
        b0, b1 = int(off[i]), int(off[i + 1])
        out.append((b0, b1, min(b1 - b0, max_seq_len)))
    return out


def attention_fwd_jvp_jagged(q, k, v, tq, tk, tv, offsets, max_seq_len,
                             causal=False, sm_scale=None, only_seqs=None):
    """Jagged forward + JVP.  q, k, tq, tk: [H, T, Dqk]; v, tv: [H, T, Dv];
    offsets: [B + 1] non-decreasing.  Sequence b attends within
    [offsets[b], offsets[b] + L_b), L_b = min(len, max_seq_len); causal
    uses in-sequence indices.  Rows of a sequence past L_b are empty rows
    (O = tO = 0, LSE = -inf); rows not covered by any sequence are NaN
    (never written).  Returns (O [H, T, Dv], tO [H, T, Dv], LSE [H, T]).
    ``only_seqs`` restricts the work to the listed sequences."""
    if torch is not None and isinstance(offsets, torch.Tensor):
        offsets = offsets.cpu().numpy()
    q, k, v, tq, tk, tv = (to_f64(x) for x in (q, k, v, tq, tk, tv))
    H, T, Dqk = q.shape
    Dv = v.shape[2]
    if sm_scale is None:
        sm_scale = default_scale(Dqk)
    O = np.full((H, T, Dv), np.nan)
    tO = np.full((H, T, Dv), np.nan)
    L = np.full((H, T), np.nan)
    for i, (b0, b1, n) in enumerate(_seq_bounds(offsets, max_seq_len)):
        if only_seqs is not None and i not in only_seqs:
            continue
        for h in range(H):
            if n > 0:
                sl = slice(b0, b0 + n)
                O[h, sl], tO[h, sl], L[h, sl] = head_fwd_jvp(
                    q[h, sl], k[h, sl], v[h, sl], tq[h, sl], tk[h, sl], tv[h, sl],
                    sm_scale, causal)
            tail = slice(b0 + n, b1)
            O[h, tail] = 0.0
            tO[h, tail] = 0.0
            L[h, tail] = NEG_INF
    return O, tO, L


def attention_fwd_jagged(q, k, v, offsets, max_seq_len, causal=False, sm_scale=None):
    """Jagged forward only: (O [H, T, Dv], LSE [H, T])."""
    if torch is not None and isinstance(offsets, torch.Tensor):
        offsets = offsets.cpu().numpy()
    q, k, v = (to_f64(x) for x in (q, k, v))
    H, T, Dqk = q.shape
    Dv = v.shape[2]
    if sm_scale is None:
        sm_scale = default_scale(Dqk)
    O = np.full((H, T, Dv), np.nan)
    L = np.full((H, T), np.nan)
    for b0, b1, n in _seq_bounds(offsets, max_seq_len):
        for h in range(H):
            if n > 0:
                sl = slice(b0, b0 + n)
                O[h, sl], L[h, sl] = head_fwd(q[h, sl], k[h, sl], v[h, sl], sm_scale, causal)
            O[h, b0 + n:b1] = 0.0
            L[h, b0 + n:b1] = NEG_INF
    return O, L
