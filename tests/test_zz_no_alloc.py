"""attn_fwd_jvp_noalloc: the entry point for callers that may not allocate
device memory (a framework that owns all device allocations, a runtime
that forbids cudaMalloc while recording work, a path with a frozen memory
budget).

Called through the C ABI twice in a row, each result must match the float64
oracle within the parity tolerances and attn_fwd_jvp's result within the
same tolerances.  The jagged case checks the fixed slot order this entry
point walks (it has no buffer for the cost-ordered work list).  A wait that
runs out of time on this path must reach the host through attn_sync_check.
A fresh process whose only calls are to this entry point must see the
device's free memory unchanged, while the allocating entry point, run
afterwards as a control, visibly allocates.

This file sorts last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh
process."""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from attention_forward_jvp_gb300 import binding, build
from attention_forward_jvp_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

O_TOL, T_TOL, L_TOL = 1e-2, 2e-2, 1e-3
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


def _compare(ref, got, what):
    """ref: float64 numpy (O, tO, LSE) or device tensors; got: device tensors."""
    ro, rto, rl = (x.float().cpu().numpy() if isinstance(x, torch.Tensor) else x for x in ref)
    go, gto, gl = (x.float().cpu().numpy() for x in got)
    assert np.isfinite(go).all() and np.isfinite(gto).all(), f"{what}: non-finite or unwritten output"
    assert not np.isnan(gl).any(), f"{what}: unwritten LSE"
    eo = np.abs(go - ro).max()
    et = np.abs(gto - rto).max()
    assert eo <= O_TOL, f"{what}: O err {eo:.3e}"
    assert et <= T_TOL * max(1.0, float(np.abs(rto).max())), f"{what}: tO err {et:.3e}"
    inf = np.isneginf(rl)
    assert np.array_equal(np.isneginf(gl), inf), f"{what}: empty-row LSE pattern"
    if (~inf).any():
        el = np.abs(gl[~inf] - rl[~inf]).max()
        assert el <= L_TOL, f"{what}: LSE err {el:.3e}"


def _case(case):
    if case == "dense_causal":
        w = Workload("na", B=1, H=3, M=333, N=333, Dqk=128, Dv=128, causal=True, tangent_std=0.5)
        inp = make_inputs(w, seed=31)
        ref = oracle.attention_fwd_jvp(inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"],
                                       causal=True, sm_scale=inp["sm_scale"])
    else:
        # lengths above and below max_seq_len, several query tiles, one token
        w = Workload("na_j", B=6, H=2, Dqk=64, Dv=64, jagged=True, max_seq_len=200,
                     max_len_draw=1, sm_scale=0.125)
        inp = make_inputs(w, seed=32, lengths=[1, 130, 64, 250, 77, 129])
        ref = oracle.attention_fwd_jvp_jagged(inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"],
                                              inp["tv"], inp["offsets"], 200, sm_scale=0.125)
    d = {n: inp[n].cuda() for n in ("q", "k", "v", "tq", "tk", "tv")}
    d["offsets"] = None if inp["offsets"] is None else inp["offsets"].cuda()
    return w, inp, d, ref


@pytest.mark.parametrize("case", ["dense_causal", "jagged"])
def test_noalloc_matches_oracle_and_attn_fwd_jvp_on_two_calls(case):
    w, inp, d, oracle_out = _case(case)
    sh, bs, out_shape, keep = binding._describe(d["q"], d["k"], d["v"], d["offsets"],
                                                inp["max_seq_len"], None, None)
    scale = float("nan") if inp["sm_scale"] is None else inp["sm_scale"]
    got = []
    for call in range(2):
        # NaN-prefilled: a row the launch does not write fails the comparison
        o = torch.full(out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        to = torch.full(out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full(out_shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc_call(d, sh, bs, w.causal, scale, o, to, lse)
        assert st == 0, f"call {call}: {binding.status_string(st)}"
        assert binding.sync_check() == 0
        _compare(oracle_out, (o, to, lse), f"{case} call {call} vs oracle")
        got.append((o, to, lse))
    ref = binding.attn_fwd_jvp(d["q"], d["k"], d["v"], d["tq"], d["tk"], d["tv"], causal=w.causal,
                               sm_scale=inp["sm_scale"], offsets=d["offsets"],
                               max_seq_len=inp["max_seq_len"])
    assert binding.sync_check() == 0
    for call, g in enumerate(got):
        _compare(ref, g, f"{case} call {call} vs attn_fwd_jvp")
    del keep


def test_noalloc_timed_out_wait_is_reported_by_sync_check():
    """The allowed failure form: the first query-tile load is skipped (a
    host-set flag), so the consumer's bounded wait runs out; the kernel
    records it in the fixed array's error word and returns, and
    attn_sync_check reports and clears it.  The next call is correct."""
    w, inp, d, oracle_out = _case("dense_causal")
    sh, bs, out_shape, keep = binding._describe(d["q"], d["k"], d["v"], None, None, None, None)
    o = torch.empty(out_shape, dtype=torch.bfloat16, device="cuda")
    to = torch.empty_like(o)
    lse = torch.empty(out_shape[:-1], dtype=torch.float32, device="cuda")
    assert binding.sync_check() == 0
    binding.set_wait_timeout_ns(100_000_000)
    binding.debug_skip_first_load(True)
    try:
        st = _noalloc_call(d, sh, bs, True, inp["sm_scale"], o, to, lse)
        status = binding.sync_check()
    finally:
        binding.debug_skip_first_load(False)
        binding.set_wait_timeout_ns(2_000_000_000)
    assert st == 0
    assert status == 5, f"expected ATTN_ERR_TIMEOUT, got {binding.status_string(status)}"
    assert binding.sync_check() == 0  # cleared
    assert _noalloc_call(d, sh, bs, True, inp["sm_scale"], o, to, lse) == 0
    assert binding.sync_check() == 0
    _compare(oracle_out, (o, to, lse), "after the timeout")
    del keep


_CHILD = r"""
import ctypes, json, os, sys
sys.path.insert(0, os.environ["ATTN_REPO_ROOT"])
from attention_forward_jvp_gb300 import binding
from attention_forward_jvp_gb300.workloads import Workload, make_inputs
import torch

L = binding.lib()
torch.cuda.init()
w = Workload("na_j", B=4, H=2, Dqk=64, Dv=64, jagged=True, max_seq_len=200, max_len_draw=1,
             sm_scale=0.125)
inp = make_inputs(w, seed=33, lengths=[5, 130, 260, 64])
d = {n: inp[n].cuda() for n in ("q", "k", "v", "tq", "tk", "tv")}
d["offsets"] = inp["offsets"].cuda()
sh, bs, out_shape, keep = binding._describe(d["q"], d["k"], d["v"], d["offsets"], 200, None, None)
o = torch.empty(out_shape, dtype=torch.bfloat16, device="cuda")
to = torch.empty_like(o)
lse = torch.empty(out_shape[:-1], dtype=torch.float32, device="cuda")
s = torch.cuda.current_stream()
p = lambda t: ctypes.c_void_p(t.data_ptr())
# the library's runtime starts (and, with eager module loading, loads its
# kernels and device arrays) at this first call, which allocates nothing
assert L.attn_sync_check(ctypes.c_void_p(s.cuda_stream)) == 0
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
for _ in range(2):
    st = L.attn_fwd_jvp_noalloc(ctypes.byref(sh), p(d["q"]), p(d["k"]), p(d["v"]), p(d["tq"]),
                                p(d["tk"]), p(d["tv"]), p(d["offsets"]), None, 0, 0.125,
                                p(o), p(to), p(lse), ctypes.c_void_p(s.cuda_stream))
    assert st == 0, st
assert L.attn_sync_check(ctypes.c_void_p(s.cuda_stream)) == 0
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
# control: the allocating entry point sets up its per-device scratch and
# this stream's work-list buffer on its first jagged call
st = L.attn_fwd_jvp(ctypes.byref(sh), p(d["q"]), p(d["k"]), p(d["v"]), p(d["tq"]), p(d["tk"]),
                    p(d["tv"]), p(d["offsets"]), None, 0, 0.125, p(o), p(to), p(lse),
                    ctypes.c_void_p(s.cuda_stream))
assert st == 0, st
assert L.attn_sync_check(ctypes.c_void_p(s.cuda_stream)) == 0
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info()[0]
print(json.dumps({"free0": free0, "free1": free1, "free2": free2}))
"""


def test_noalloc_allocates_no_device_memory_in_a_fresh_process():
    env = dict(os.environ, ATTN_REPO_ROOT=ROOT, CUDA_MODULE_LOADING="EAGER")
    r = subprocess.run([sys.executable, "-c", _CHILD], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    m = json.loads(r.stdout.strip().splitlines()[-1])
    if m["free2"] >= m["free1"]:
        pytest.skip("the free-memory reading does not show the control's allocation on this driver")
    assert m["free1"] == m["free0"], (
        f"device free memory changed by {m['free0'] - m['free1']} bytes across two allocation-free calls")
