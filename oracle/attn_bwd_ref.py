"""Float64 CPU oracle for the attention backward pass (dQ, dK, dV).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests and the benchmark's
CPU legs may import this module.  It shares no code with the CUDA path; it
reuses the forward oracle's scores / valid-set / softmax steps (attn_ref)
and materialises every intermediate, in float64, one head at a time.

Given the forward of one head (S = s Q K^T + bias, P = softmax over the
valid keys, O = P V) and the gradient dO of a loss with respect to O:

  dV    = P^T dO
  dP    = dO V^T
  Delta = rowsum(dO o O)              (= rowsum(P o dP))
  dS    = P o (dP - Delta)            (the softmax backward)
  dQ    = s dS K
  dK    = s dS^T Q
  (the bias gets no gradient here; empty rows have P = 0 and add nothing)

Sources (the pages; code, so each step is a code step):
  * the Triton fused-attention tutorial backward ("_attn_bwd_preprocess":
    ``delta = sum(o * do, axis=1)``; "_attn_bwd_dkdv": ``pT = exp2(qkT - m)``
    from the stored log-sum-exp, ``dv += pT do``, ``dpT = v do^T``,
    ``dsT = pT * (dpT - Di)``, ``dk += dsT q``; "_attn_bwd_dq":
    ``ds = p * (dp - Di)``, ``dq += ds k``; dq and dk carry the softmax
    scale);
  * "flash_attention.py" (triton_flashattn) "_attn_bwd_preprocess" and
    "_attn_bwd_dkdv_inner" / "_attn_bwd_dq_inner" (the same steps with
    unequal head dims and per-tensor strides);
  * FBGEMM's jagged backward ("_multi_head_jagged_flash_attention_bwd_kernel":
    ``ds = p * (dp - delta)``) for the jagged layout.
"""
from __future__ import annotations

import numpy as np

from .attn_ref import (_bh, _seq_bounds, default_scale, scores, softmax_rows, to_f64,
                       valid_keys)


def head_bwd(q, k, v, do, sm_scale, causal=False, bias=None, mask=None, row_index=None):
    """Backward of one head, float64.  q: [m, Dqk]; k: [n, Dqk]; v: [n, Dv];
    do: [m, Dv]; bias [m, n] or None; mask [m, n] bool or None.
    Returns (dQ [m, Dqk], dK [n, Dqk], dV [n, Dv], Delta [m])."""
    m, n = q.shape[0], k.shape[0]
    ok = valid_keys(m, n, causal, row_index, mask)
    p, _ = softmax_rows(scores(q, k, sm_scale, bias), ok)
    o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    delta = (do * o).sum(axis=1)
    ds = p * (dp - delta[:, None])
    dq = sm_scale * (ds @ k)
    dk = sm_scale * (ds.T @ q)
    return dq, dk, dv, delta


def attention_bwd(q, k, v, do, causal=False, sm_scale=None, bias=None, mask=None):
    """Dense backward.  q: [B, H, M, Dqk]; k: [B, H, N, Dqk]; v: [B, H, N, Dv];
    do: [B, H, M, Dv]; bias / mask as in the forward oracle.  Returns
    float64 (dQ, dK, dV, Delta) shaped like q, k, v and [B, H, M]."""
    q, k, v, do = (to_f64(x) for x in (q, k, v, do))
    bias = to_f64(bias)
    mask = None if mask is None else (to_f64(mask) != 0)
    B, H, M, _ = q.shape
    N = k.shape[2]
    if sm_scale is None:
        sm_scale = default_scale(q.shape[3])
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    Dl = np.zeros((B, H, M))
    for b in range(B):
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h], Dl[b, h] = head_bwd(
                q[b, h], k[b, h], v[b, h], do[b, h], sm_scale, causal,
                _bh(bias, b, h, (M, N)), _bh(mask, b, h, (M, N)))
    return dQ, dK, dV, Dl


def attention_bwd_jagged(q, k, v, do, offsets, max_seq_len, causal=False, sm_scale=None):
    """Jagged backward over [H, T, D] tensors with offsets[B + 1]: sequence b
    attends within its first min(len, max_seq_len) tokens; tokens past that
    (and tokens of no sequence) get zero gradients."""
    try:
        import torch
        if isinstance(offsets, torch.Tensor):
            offsets = offsets.cpu().numpy()
    except Exception:  # pragma: no cover
        pass
    q, k, v, do = (to_f64(x) for x in (q, k, v, do))
    H, T, Dqk = q.shape
    if sm_scale is None:
        sm_scale = default_scale(Dqk)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    Dl = np.zeros((H, T))
    for b0, _b1, n in _seq_bounds(offsets, max_seq_len):
        if n == 0:
            continue
        sl = slice(b0, b0 + n)
        for h in range(H):
            dQ[h, sl], dK[h, sl], dV[h, sl], Dl[h, sl] = head_bwd(
                q[h, sl], k[h, sl], v[h, sl], do[h, sl], sm_scale, causal)
    return dQ, dK, dV, Dl
