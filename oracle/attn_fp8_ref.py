"""Float64 CPU oracle for the FP8 (e5m2) attention forward.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests and the benchmark's
CPU legs may import this module.  It shares no code with the CUDA path.

The FP8 path is an approximation of attention, so the oracle takes the
algorithm's steps in the order of the Triton fused-attention tutorial with
JVP ("_06_fused_attention_blockptr_jvp.py"): in `_attn_fwd_inner_tma` the
row sum `l` is taken from the fp32 weights `p = exp2(qk - m)` and only then
is `p` cast to the input dtype (`p = p.to(dtype)`, float8e5) for the `p v`
dot; `JVPAttn.forward` allocates `o = torch.empty_like(q)`, so the
normalised output is stored in e5m2 as well; V arrives transposed.
Everything else is the plain definition in float64 on the (exact) e5m2
input values:

  S   = s Q K^T                       (causal: -inf for j > i)
  m   = max_j S_ij,   p = exp(S - m),   l = sum_j p
  O   = e5m2( (e5m2(p) V) / l )
  LSE = m + log l                     (no rounding)
  empty rows: O = 0, LSE = -inf

e5m2 rounding (one sign, five exponent and two mantissa bits, round to
nearest even) is torch's float8_e5m2 conversion, a library primitive used
as a step; tests/test_oracle_fp8.py pins it to hand-derived values.
"""
from __future__ import annotations

import numpy as np
import torch

from .attn_ref import default_scale, scores, to_f64, valid_keys


def round_e5m2(x) -> np.ndarray:
    """Nearest e5m2 value of each float64 element (ties to even)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float64))
    return t.to(torch.float8_e5m2).to(torch.float64).numpy()


def head_fwd_e5m2(q, k, v, sm_scale, causal=False):
    """One head.  q [m, D], k [n, D], v [n, Dv] (float64 values of e5m2
    inputs).  Returns (O [m, Dv] on the e5m2 grid, LSE [m])."""
    m_rows, n = q.shape[0], k.shape[0]
    ok = valid_keys(m_rows, n, causal, None, None)
    s = np.where(ok, scores(q, k, sm_scale, None), -np.inf)
    mx = s.max(axis=1) if n > 0 else np.full(m_rows, -np.inf)
    empty = ~np.isfinite(mx)
    mx_safe = np.where(empty, 0.0, mx)
    p = np.where(ok, np.exp(s - mx_safe[:, None]), 0.0)
    l = p.sum(axis=1)
    o = (round_e5m2(p) @ v) / np.where(empty, 1.0, l)[:, None]
    o = np.where(empty[:, None], 0.0, round_e5m2(o))
    lse = np.where(empty, -np.inf, mx_safe + np.log(np.where(empty, 1.0, l)))
    return o, lse


def attention_fwd_e5m2(q, k, v, causal=False, sm_scale=None):
    """Dense FP8 forward.  q [B, H, M, D], k [B, H, N, D], v [B, H, N, Dv]
    (torch float8_e5m2 or float64 of such values; V in its natural,
    untransposed orientation).  Returns float64 (O, LSE)."""
    q, k, v = (to_f64(x) for x in (q, k, v))
    B, H, M, D = q.shape
    if sm_scale is None:
        sm_scale = default_scale(D)
    O = np.zeros((B, H, M, v.shape[3]))
    L = np.zeros((B, H, M))
    for b in range(B):
        for h in range(H):
            O[b, h], L[b, h] = head_fwd_e5m2(q[b, h], k[b, h], v[b, h], sm_scale, causal)
    return O, L


def e5m2_bound_terms(q, k, v, sm_scale, causal=False):
    """Float64 quantities the e5m2 roundings are bounded by, per output
    element of one head: B = sum_j w_j |V_j| (w the exact softmax weights)
    and the exact output O = sum_j w_j V_j.  Weights w_j rounded to
    w_j (1 + d_j), |d_j| <= 2^-3, with the row sum of the unrounded weights
    (the tutorial's order), move the output by at most 2^-3 B."""
    m_rows, n = q.shape[0], k.shape[0]
    ok = valid_keys(m_rows, n, causal, None, None)
    if n == 0:
        z = np.zeros((m_rows, v.shape[1]))
        return z, z
    s = np.where(ok, scores(q, k, sm_scale, None), -np.inf)
    mx = s.max(axis=1)
    empty = ~np.isfinite(mx)
    p = np.where(ok, np.exp(s - np.where(empty, 0.0, mx)[:, None]), 0.0)
    w = p / np.where(empty, 1.0, p.sum(axis=1))[:, None]
    return w @ np.abs(v), w @ v
