"""Seeded synthetic workloads for attention forward + JVP.

This module only draws random inputs and describes shapes. It holds none of
the attention arithmetic, so both the CUDA path and the float64 oracle can be
fed from it without sharing any computation.

Recipe (all on the CPU, torch generator seeded per call):
  * draw order q, k, v, tq, tk, tv, then the fp32 bias; for the jagged
    workload the sequence lengths are drawn first, because the packed
    ``[H, T, D]`` shapes depend on them;
  * every value is ``randn`` in fp32 times the stated standard deviation,
    then cast to bf16 with round-to-nearest-even;
  * the key-padding mask keeps the first ``mask_keep`` keys of every batch
    entry and is stored as ``uint8 [B, 1, 1, N]`` (broadcast over heads and
    query rows, 1 = attend).

Workload names follow what they are, not where they came from:
  tiny        B1 H2  N128  D64   non-causal
  noncausal   B4 H16 N1024 D64   non-causal
  causal      B2 H16 N4096 D128  causal, tangents N(0, 0.5^2)
  jagged      64 sequences, lengths U{1..1024}, H8 D64, packed [H, T, D]
  bias_mask   B2 H8 M=N=2048 Dqk128 Dv64, fp32 bias N(0,1), keys >= 1536 masked
  causal_d256 B2 H16 N4096 Dqk=Dv=256 causal, tangents N(0, 0.5^2)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    M: int = 0            # dense query length (jagged: max_seq_len)
    N: int = 0            # dense key length (jagged: max_seq_len)
    Dqk: int = 64
    Dv: int = 64
    causal: bool = False
    jagged: bool = False
    max_seq_len: int = 0  # jagged only
    max_len_draw: int = 0  # jagged only: lengths ~ U{1..max_len_draw}
    input_std: float = 1.0
    tangent_std: float = 1.0
    sm_scale: Optional[float] = None   # None = Dqk ** -0.5
    bias: bool = False
    mask_keep: Optional[int] = None    # keys j < mask_keep attend (key padding)

    @property
    def scale(self) -> float:
        return self.sm_scale if self.sm_scale is not None else self.Dqk ** -0.5

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, H=2, M=128, N=128, Dqk=64, Dv=64, sm_scale=1.0 / 8),
    "noncausal": Workload("noncausal", B=4, H=16, M=1024, N=1024, Dqk=64, Dv=64, sm_scale=1.0 / 8),
    "causal": Workload("causal", B=2, H=16, M=4096, N=4096, Dqk=128, Dv=128, causal=True,
                       tangent_std=0.5, sm_scale=1.0 / math.sqrt(128)),
    "jagged": Workload("jagged", B=64, H=8, M=1024, N=1024, Dqk=64, Dv=64, jagged=True,
                       max_seq_len=1024, max_len_draw=1024, sm_scale=1.0 / 8),
    "bias_mask": Workload("bias_mask", B=2, H=8, M=2048, N=2048, Dqk=128, Dv=64, bias=True,
                          mask_keep=1536),
    # head dim 256 with tangents (the widest head dim the kernels accept);
    # the causal workload's shape and distributions otherwise
    "causal_d256": Workload("causal_d256", B=2, H=16, M=4096, N=4096, Dqk=256, Dv=256, causal=True,
                            tangent_std=0.5, sm_scale=1.0 / 16),
}


def _randn(g: torch.Generator, shape, std: float) -> torch.Tensor:
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def make_inputs(w: Workload, seed: int = 0, lengths: Optional[list] = None) -> dict:
    """Draw the inputs of workload ``w`` on the CPU.

    Returns a dict with bf16 tensors ``q, k, v, tq, tk, tv`` (dense
    ``[B, H, M|N, D]``, jagged ``[H, T, D]``), optional ``bias`` (fp32
    ``[B, H, M, N]``), optional ``mask`` (uint8 ``[B, 1, 1, N]``), optional
    int32 ``offsets`` ``[B + 1]`` and the scalars ``sm_scale``, ``causal``,
    ``max_seq_len``.  ``lengths`` overrides the drawn jagged lengths.
    """
    g = torch.Generator().manual_seed(seed)
    out = {"workload": w, "sm_scale": w.scale, "causal": w.causal,
           "bias": None, "mask": None, "offsets": None, "max_seq_len": None}
    if w.jagged:
        if lengths is None:
            lens = torch.randint(1, w.max_len_draw + 1, (w.B,), generator=g, dtype=torch.int64)
        else:
            lens = torch.tensor(lengths, dtype=torch.int64)
            assert lens.numel() == w.B
        offsets = torch.zeros(w.B + 1, dtype=torch.int64)
        offsets[1:] = torch.cumsum(lens, 0)
        T = int(offsets[-1])
        qs = (w.H, T, w.Dqk)
        ks = (w.H, T, w.Dqk)
        vs = (w.H, T, w.Dv)
        out["offsets"] = offsets.to(torch.int32)
        out["max_seq_len"] = w.max_seq_len
    else:
        qs = (w.B, w.H, w.M, w.Dqk)
        ks = (w.B, w.H, w.N, w.Dqk)
        vs = (w.B, w.H, w.N, w.Dv)
    out["q"] = _randn(g, qs, w.input_std)
    out["k"] = _randn(g, ks, w.input_std)
    out["v"] = _randn(g, vs, w.input_std)
    out["tq"] = _randn(g, qs, w.tangent_std)
    out["tk"] = _randn(g, ks, w.tangent_std)
    out["tv"] = _randn(g, vs, w.tangent_std)
    if w.bias:
        out["bias"] = torch.randn((w.B, w.H, w.M, w.N), generator=g, dtype=torch.float32)
    if w.mask_keep is not None:
        m = torch.zeros((w.B, 1, 1, w.N), dtype=torch.uint8)
        m[..., : w.mask_keep] = 1
        out["mask"] = m
    return out


def flops_fwd_jvp(w: Workload, offsets: Optional[torch.Tensor] = None) -> float:
    """Algorithmic FLOPs of forward + JVP: six matmuls per score element,
    three QK-shaped (2*Dqk each) and three PV-shaped (2*Dv each), halved
    for causal attention (the FLOP rule of the JVP benchmark in
    "Flash Attention v2 with JVP", ``bench_flash_attention``)."""
    per_elem = 6.0 * (w.Dqk + w.Dv)
    if w.jagged:
        assert offsets is not None
        lens = (offsets[1:] - offsets[:-1]).clamp(max=w.max_seq_len).to(torch.float64)
        n_elem = float((lens * lens).sum()) * w.H
    else:
        n_elem = float(w.B * w.H * w.M * w.N)
    f = per_elem * n_elem
    if w.causal:
        f *= 0.5
    return f


def flops_fwd(w: Workload, offsets: Optional[torch.Tensor] = None) -> float:
    """Forward only: two matmuls per score element (QK and PV)."""
    return flops_fwd_jvp(w, offsets) / 3.0


def min_hbm_bytes(w: Workload, inputs: dict, jvp: bool = True) -> int:
    """Bytes that must cross HBM at least once: every input read, every
    output written once."""
    n = 0
    names = ("q", "k", "v", "tq", "tk", "tv") if jvp else ("q", "k", "v")
    for nm in names:
        n += inputs[nm].numel() * 2
    q, v = inputs["q"], inputs["v"]
    rows = q.numel() // w.Dqk
    n += rows * w.Dv * 2 * (2 if jvp else 1)   # O (and tO)
    n += rows * 4                               # LSE
    if inputs.get("bias") is not None:
        n += inputs["bias"].numel() * 4
    if inputs.get("mask") is not None:
        n += inputs["mask"].numel()
    return n


def make_bwd_inputs(w: Workload, seed: int = 0, lengths: Optional[list] = None) -> dict:
    """Inputs of the backward for workload ``w``: bf16 ``q, k, v`` and the
    output gradient ``do`` (dense ``[B, H, M|N, D]``, jagged ``[H, T, D]``),
    drawn in that order (``randn`` times ``input_std``; ``do`` at std 1),
    after the jagged lengths (``lengths`` overrides them), plus
    ``sm_scale``, ``causal``, ``offsets``, ``max_seq_len``.  The forward's O
    and LSE are not drawn: each side computes its own."""
    g = torch.Generator().manual_seed(seed)
    out = {"workload": w, "sm_scale": w.scale, "causal": w.causal, "offsets": None, "max_seq_len": None}
    if w.jagged:
        if lengths is None:
            lens = torch.randint(1, w.max_len_draw + 1, (w.B,), generator=g, dtype=torch.int64)
        else:
            lens = torch.tensor(lengths, dtype=torch.int64)
            assert lens.numel() == w.B
        offsets = torch.zeros(w.B + 1, dtype=torch.int64)
        offsets[1:] = torch.cumsum(lens, 0)
        T = int(offsets[-1])
        qs, ks, vs = (w.H, T, w.Dqk), (w.H, T, w.Dqk), (w.H, T, w.Dv)
        out["offsets"] = offsets.to(torch.int32)
        out["max_seq_len"] = w.max_seq_len
    else:
        qs, ks, vs = (w.B, w.H, w.M, w.Dqk), (w.B, w.H, w.N, w.Dqk), (w.B, w.H, w.N, w.Dv)
    out["q"] = _randn(g, qs, w.input_std)
    out["k"] = _randn(g, ks, w.input_std)
    out["v"] = _randn(g, vs, w.input_std)
    out["do"] = _randn(g, qs[:-1] + (w.Dv,), 1.0)
    return out


def score_elements(w: Workload, offsets: Optional[torch.Tensor] = None) -> float:
    """Score elements of the workload before the causal halving: B H M N
    dense, H sum_b min(L_b, max_seq_len)^2 jagged."""
    if w.jagged:
        assert offsets is not None
        lens = (offsets[1:] - offsets[:-1]).clamp(max=w.max_seq_len).to(torch.float64)
        return float((lens * lens).sum()) * w.H
    return float(w.B * w.H * w.M * w.N)


def flops_bwd(w: Workload, offsets: Optional[torch.Tensor] = None) -> float:
    """Algorithmic FLOPs of the backward: five matmuls per score element
    (S = Q K^T, dP = dO V^T, dV = P^T dO, dQ = dS K, dK = dS^T Q), halved
    for causal attention -- 2.5 times the forward, the rule of the
    fused-attention tutorial's benchmark.  Kernels that recompute a product
    do not get credit for it."""
    f = 2.0 * (3 * w.Dqk + 2 * w.Dv) * score_elements(w, offsets)
    if w.causal:
        f *= 0.5
    return f


def min_hbm_bytes_bwd(w: Workload, rows: Optional[int] = None) -> int:
    """Bytes the backward must move at least once: q, k, v, o, do, lse read;
    dq, dk, dv written (all 16-bit but lse); Delta written and read (fp32).
    ``rows``: jagged H T (query rows = key rows)."""
    if rows is not None:
        rows_q = rows_k = rows
    else:
        rows_q, rows_k = w.B * w.H * w.M, w.B * w.H * w.N
    n = 2 * (rows_q * w.Dqk + rows_k * (w.Dqk + w.Dv) + 2 * rows_q * w.Dv)
    n += 4 * rows_q                          # lse
    n += 2 * (rows_q * w.Dqk + rows_k * (w.Dqk + w.Dv))
    n += 2 * 4 * rows_q                      # Delta out + in
    return n


def make_f8_inputs(w: Workload, seed: int = 0) -> dict:
    """Inputs of the FP8 forward for dense workload ``w``: ``q, k, v`` drawn
    as ``randn`` fp32 times ``input_std`` in that order, rounded to
    float8_e5m2 (v in its natural [B, H, N, Dv] orientation), and ``vt``,
    v transposed to [B, H, Dv, N] and made contiguous (the FP8 layout)."""
    assert not w.jagged and w.Dqk == w.Dv
    g = torch.Generator().manual_seed(seed)

    def draw(shape):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if w.input_std != 1.0:
            x = x * w.input_std
        return x.to(torch.float8_e5m2)

    q = draw((w.B, w.H, w.M, w.Dqk))
    k = draw((w.B, w.H, w.N, w.Dqk))
    v = draw((w.B, w.H, w.N, w.Dv))
    return {"workload": w, "sm_scale": w.scale, "causal": w.causal, "q": q, "k": k, "v": v,
            "vt": v.transpose(-1, -2).contiguous()}
