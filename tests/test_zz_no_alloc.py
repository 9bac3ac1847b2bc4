"""attn_fwd_jvp_noalloc: the entry point for callers that may not allocate
device memory (a framework that owns all device allocations, a runtime
that forbids cudaMalloc while recording work, a path with a frozen memory
budget).  Called through the C ABI twice in a row; each result must match
attn_fwd_jvp's within the parity tolerances.  This file sorts last so that
a run stopping at its first failure has already run every other test; it
also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from attention_forward_jvp_gb300 import binding, build
from attention_forward_jvp_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

O_TOL, T_TOL, L_TOL = 1e-2, 2e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.lib()


def _noalloc_call(d, sh, bs, causal, scale, o, to, lse):
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    st = binding.lib().attn_fwd_jvp_noalloc(
        ctypes.byref(sh), p(d["q"]), p(d["k"]), p(d["v"]), p(d["tq"]), p(d["tk"]), p(d["tv"]),
        p(d.get("offsets")), ctypes.byref(bs) if bs is not None else None, 1 if causal else 0,
        float(scale), p(o), p(to), p(lse), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _compare(ref, got):
    (ro, rto, rl), (go, gto, gl) = ref, got
    ro, rto, go, gto = (x.float().cpu().numpy() for x in (ro, rto, go, gto))
    rl, gl = rl.cpu().numpy(), gl.cpu().numpy()
    assert np.isfinite(go).all() and np.isfinite(gto).all()
    assert np.abs(go - ro).max() <= O_TOL
    assert np.abs(gto - rto).max() <= T_TOL * max(1.0, float(np.abs(rto).max()))
    inf = np.isneginf(rl)
    assert np.array_equal(np.isneginf(gl), inf)
    if (~inf).any():
        assert np.abs(gl[~inf] - rl[~inf]).max() <= L_TOL


@pytest.mark.parametrize("case", ["dense_causal", "jagged"])
def test_noalloc_matches_attn_fwd_jvp_on_two_calls(case):
    if case == "dense_causal":
        w = Workload("na", B=1, H=3, M=333, N=333, Dqk=128, Dv=128, causal=True, tangent_std=0.5)
        inp = make_inputs(w, seed=31)
    else:
        w = Workload("na_j", B=5, H=2, Dqk=64, Dv=64, jagged=True, max_seq_len=200,
                     max_len_draw=1, sm_scale=0.125)
        inp = make_inputs(w, seed=32, lengths=[1, 130, 64, 250, 77])
    d = {n: inp[n].cuda() for n in ("q", "k", "v", "tq", "tk", "tv")}
    d["offsets"] = None if inp["offsets"] is None else inp["offsets"].cuda()
    kw = dict(causal=w.causal, sm_scale=inp["sm_scale"], offsets=d["offsets"],
              max_seq_len=inp["max_seq_len"])
    ref = binding.attn_fwd_jvp(d["q"], d["k"], d["v"], d["tq"], d["tk"], d["tv"], **kw)
    assert binding.sync_check() == 0
    sh, bs, out_shape, keep = binding._describe(d["q"], d["k"], d["v"], d["offsets"],
                                                inp["max_seq_len"], None, None)
    scale = float("nan") if inp["sm_scale"] is None else inp["sm_scale"]
    for call in range(2):
        o = torch.full(out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        to = torch.full(out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full(out_shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc_call(d, sh, bs, w.causal, scale, o, to, lse)
        assert st == 0, f"call {call}: {binding.status_string(st)}"
        torch.cuda.synchronize()
        _compare(ref, (o, to, lse))
    del keep
