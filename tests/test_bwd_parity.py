"""GPU parity of the attention backward (dQ, dK, dV, Delta) through the C
ABI against the float64 oracle (oracle.attention_bwd / head_bwd).

The chain under test is the one a user runs: the library's forward writes
O and LSE, the library's backward takes them with dO.  The oracle takes
only q, k, v, dO from the seeded generator and recomputes everything.

Tolerance (derived from the arithmetic; no published one covers the
backward): P and dS enter the tensor-core products as 16-bit values
(relative rounding 2^-9 for bf16) and O comes from the forward in bf16, the
same error sources as the forward's tangent output, so each gradient G
must satisfy max|G - G_oracle| <= 2e-2 * max(1, ||G_oracle||_inf) and
Delta max|err| <= 1e-2 * max(1, ||Delta_oracle||_inf).
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_jvp_gb300 import binding, build
from attention_forward_jvp_gb300.workloads import WORKLOADS, Workload, make_bwd_inputs

pytestmark = pytest.mark.gpu

G_TOL = 2e-2
D_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.lib()


def run_gpu_bwd(inp, f16=False):
    cast = (lambda t: t.float().half()) if f16 else (lambda t: t)
    q, k, v, do = (cast(inp[n]).cuda() for n in ("q", "k", "v", "do"))
    kw = dict(causal=inp["causal"], sm_scale=inp["sm_scale"])
    for n in ("bias", "mask"):
        if inp.get(n) is not None:
            kw[n] = inp[n].cuda()
    o, lse = binding.attn_fwd(q, k, v, **kw)
    dq, dk, dv, delta = binding.attn_bwd(q, k, v, o, lse, do, **kw)
    assert binding.sync_check() == 0
    return tuple(t.float().cpu().numpy() for t in (dq, dk, dv, delta))


def oracle_bwd(inp, f16=False):
    cast = (lambda t: t.float().half()) if f16 else (lambda t: t)
    return oracle.attention_bwd(*(cast(inp[n]) for n in ("q", "k", "v", "do")),
                                causal=inp["causal"], sm_scale=inp["sm_scale"],
                                bias=inp.get("bias"), mask=inp.get("mask"))


def assert_grads_close(got, ref, what=""):
    errs = []
    for name, g, r in zip(("dQ", "dK", "dV"), got[:3], ref[:3]):
        assert g.shape == r.shape, f"{what}: {name} shape {g.shape} vs {r.shape}"
        assert np.isfinite(g).all(), f"{what}: non-finite {name}"
        e = float(np.abs(g - r).max()) if g.size else 0.0
        scale = max(1.0, float(np.abs(r).max()) if r.size else 0.0)
        assert e <= G_TOL * scale, f"{what}: {name} err {e:.3e} (scale {scale:.2f})"
        errs.append(e / scale)
    g, r = got[3], ref[3]
    e = float(np.abs(g - r).max()) if g.size else 0.0
    scale = max(1.0, float(np.abs(r).max()) if r.size else 0.0)
    assert e <= D_TOL * scale, f"{what}: Delta err {e:.3e} (scale {scale:.2f})"
    return errs


def _w(**kw):
    base = dict(name="bwd", B=1, H=2, M=256, N=256, Dqk=64, Dv=64)
    base.update(kw)
    return Workload(**base)


CASES = [
    # name, workload
    ("nc_d64", _w(M=384, N=384)),
    ("causal_d64", _w(M=320, N=320, causal=True)),
    ("nc_d128", _w(M=256, N=320, Dqk=128, Dv=128)),
    ("causal_d128", _w(M=448, N=448, Dqk=128, Dv=128, causal=True)),
    ("cross_ragged", _w(B=2, H=1, M=200, N=333)),
    ("short_q", _w(M=1, N=515)),
    ("short_k", _w(M=300, N=1)),
    ("tiny_causal", _w(M=5, N=5, causal=True)),
    ("d16", _w(M=200, N=260, Dqk=16, Dv=16)),
    ("d32_causal", _w(M=257, N=257, Dqk=32, Dv=32, causal=True)),
    ("scale_std2", _w(M=256, N=384, input_std=2.0, sm_scale=0.2)),
    # unequal head dims (the flash_attention.py backward's Dqk != Dv)
    ("dqk128_dv64_causal", _w(M=320, N=320, Dqk=128, Dv=64, causal=True)),
    ("dqk64_dv128", _w(M=200, N=333, Dqk=64, Dv=128)),
    ("dqk32_dv128_causal", _w(M=257, N=257, Dqk=32, Dv=128, causal=True)),
    ("dqk128_dv16", _w(M=130, N=260, Dqk=128, Dv=16)),
]


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_bwd_parity(name, w):
    inp = make_bwd_inputs(w, seed=7)
    assert_grads_close(run_gpu_bwd(inp), oracle_bwd(inp), what=name)


@pytest.mark.parametrize("name,w", [CASES[1], CASES[2], CASES[11]], ids=["causal_d64", "nc_d128", "dqk128_dv64"])
def test_bwd_parity_f16(name, w):
    inp = make_bwd_inputs(w, seed=8)
    assert_grads_close(run_gpu_bwd(inp, f16=True), oracle_bwd(inp, f16=True), what=name + "_f16")


def test_bwd_empty_sides():
    # no queries: dK = dV = 0; no keys: dQ = 0
    for M, N in ((0, 200), (130, 0)):
        w = _w(M=M, N=N)
        inp = make_bwd_inputs(w, seed=3)
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
        o = torch.zeros_like(do)
        lse = torch.full((w.B, w.H, w.M), float("-inf"), device="cuda")
        dq, dk, dv, delta = (torch.full_like(t, 7.0) for t in (q, k, v, lse))
        binding.attn_bwd(q, k, v, o, lse, do, out=(dq, dk, dv, delta))
        assert binding.sync_check() == 0
        assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0)
        assert torch.all(delta == 0)


def test_bwd_unsupported_configs():
    inp = make_bwd_inputs(_w(M=128, N=128, Dqk=64, Dv=256), seed=1)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    lse = torch.zeros(1, 2, 128, device="cuda")
    with pytest.raises(binding.AttnError) as e:
        binding.attn_bwd(q, k, v, do, lse, do)
    assert e.value.status == 2  # Dv = 256


@pytest.mark.parametrize("name", ["causal", "noncausal"])
def test_bwd_full_size_whole_output(name):
    # the benchmark's backward shapes (B2 H16 N4096 D128 causal, B4 H16 N1024
    # D64 non-causal), outputs prefilled with NaN so that a unit the
    # persistent schedule skipped would show; every head whole against the
    # oracle, and at every head the identity sum_j dK_j = 0 (adding one
    # vector to every key leaves each row's softmax unchanged)
    w = WORKLOADS[name]
    inp = make_bwd_inputs(w, seed=0)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    kw = dict(causal=inp["causal"], sm_scale=inp["sm_scale"])
    o, lse = binding.attn_fwd(q, k, v, **kw)
    out = tuple(torch.full_like(t, float("nan")) for t in (q, k, v, lse))
    binding.attn_bwd(q, k, v, o, lse, do, out=out, **kw)
    assert binding.sync_check() == 0
    dq, dk, dv, delta = (t.float().cpu().numpy() for t in out)
    for t in (dq, dk, dv, delta):
        assert not np.isnan(t).any(), f"{name}: unwritten gradient rows"
    assert_grads_close((dq, dk, dv, delta), oracle_bwd(inp), what=name)
    col = np.abs(dk.astype(np.float64).sum(axis=2))
    scale = np.abs(dk).max()
    assert col.max() <= 2e-2 * max(1.0, scale) * 8, f"sum_j dK_j = {col.max():.3e}"


def test_bwd_stages_match_one_call():
    # Delta, the dQ pass and the dK / dV pass launched one by one give
    # bitwise the results of one attn_bwd call
    inp = make_bwd_inputs(_w(M=300, N=300, causal=True), seed=11)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    kw = dict(causal=True, sm_scale=inp["sm_scale"])
    o, lse = binding.attn_fwd(q, k, v, **kw)
    ref = binding.attn_bwd(q, k, v, o, lse, do, **kw)
    out = tuple(torch.full_like(t, 3.0) for t in ref)
    for sg in (binding.BWD_DELTA, binding.BWD_DKDV, binding.BWD_DQ):
        binding.attn_bwd(q, k, v, o, lse, do, out=out, stages=sg, **kw)
    assert binding.sync_check() == 0
    for a, b in zip(ref, out):
        assert torch.equal(a, b)


JAGGED_LENS = [3, 64, 130, 257, 1, 0, 300, 128]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128, 32, (128, 64)])
def test_bwd_jagged(causal, D):
    # lengths around the tile sizes, an empty sequence and two sequences
    # past max_seq_len = 256 (their capped tokens get zero gradients)
    dqk, dv = D if isinstance(D, tuple) else (D, D)
    w = Workload("jb", B=len(JAGGED_LENS), H=2, Dqk=dqk, Dv=dv, jagged=True, max_seq_len=256,
                 max_len_draw=1, causal=causal)
    inp = make_bwd_inputs(w, seed=21, lengths=JAGGED_LENS)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    off = inp["offsets"].cuda()
    kw = dict(causal=causal, sm_scale=inp["sm_scale"], offsets=off, max_seq_len=256)
    o, lse = binding.attn_fwd(q, k, v, **kw)
    dq, dk, dv, delta = binding.attn_bwd(q, k, v, o, lse, do, **kw)
    assert binding.sync_check() == 0
    got = tuple(t.float().cpu().numpy() for t in (dq, dk, dv, delta))
    ref = oracle.attention_bwd_jagged(inp["q"], inp["k"], inp["v"], inp["do"], inp["offsets"], 256,
                                      causal=causal, sm_scale=inp["sm_scale"])
    assert_grads_close(got, ref, what=f"jagged D{D} causal={causal}")
    # capped tokens: exactly zero
    offs = inp["offsets"].numpy()
    for b, L in enumerate(JAGGED_LENS):
        if L > 256:
            for g in got[:3]:
                assert np.all(g[:, offs[b] + 256:offs[b + 1]] == 0)


# ------------------------------------------------------ bias / mask backward
# The same bias and mask go to the forward and the backward (the pages'
# bias backward, "flash_attention.py" _attn_bwd_dkdv_inner /
# _attn_bwd_dq_inner, without the bias gradient).
def _bias_mask(B, H, M, N, kind, seed):
    g = torch.Generator().manual_seed(seed)
    bias = mask = None
    if "bias" in kind:
        bias = torch.randn((B, H, M, N), generator=g)
    if "rowmask" in kind:
        mask = (torch.rand((B, 1, M, N), generator=g) < 0.7).to(torch.uint8)
        mask[0, 0, 3, :] = 0  # a fully masked row: LSE = -inf, no gradient through it
    if "keymask" in kind:
        mask = torch.ones((B, 1, 1, N), dtype=torch.uint8)
        mask[..., N - N // 4:] = 0
        mask[-1, ..., 5] = 0
    if "headbias" in kind:
        bias = torch.randn((1, H, 1, N), generator=g)  # broadcast over batch and rows
    return bias, mask


BIAS_CASES = [
    ("bias", dict(M=256, N=320, Dqk=64, Dv=64), "bias"),
    ("bias_rowmask", dict(M=200, N=333, Dqk=128, Dv=64), "bias+rowmask"),
    ("causal_bias_keymask", dict(M=384, N=384, Dqk=128, Dv=128, causal=True), "bias+keymask"),
    ("keymask_only", dict(M=260, N=300, Dqk=64, Dv=128), "keymask"),
    ("headbias_broadcast", dict(M=190, N=257, Dqk=32, Dv=64), "headbias"),
]


@pytest.mark.parametrize("name,shape,kind", BIAS_CASES, ids=[c[0] for c in BIAS_CASES])
def test_bwd_with_bias_and_mask(name, shape, kind):
    w = _w(B=2, **shape)
    inp = make_bwd_inputs(w, seed=71)
    inp["bias"], inp["mask"] = _bias_mask(2, w.H, w.M, w.N, kind, seed=72)
    assert_grads_close(run_gpu_bwd(inp), oracle_bwd(inp), what=name)


def test_bwd_with_bias_fp16():
    w = _w(B=1, M=200, N=264, Dqk=64, Dv=64)
    inp = make_bwd_inputs(w, seed=73)
    inp["bias"], inp["mask"] = _bias_mask(1, w.H, w.M, w.N, "bias+rowmask", seed=74)
    assert_grads_close(run_gpu_bwd(inp, f16=True), oracle_bwd(inp, f16=True), what="fp16 bias")



def _random_bwd_case(rng):
    """One seeded draw over the backward's supported set: head dims for Q / K
    and V independently in {16, 32, 64, 128}; dense (causal, cross-attention
    lengths, bias and / or key mask) or jagged (lengths around tile edges
    and past the cap); bf16 or fp16."""
    dims = [16, 32, 64, 128]
    dqk, dv = int(rng.choice(dims)), int(rng.choice(dims))
    causal = rng.random() < 0.4
    if rng.random() < 0.3:
        nb = int(rng.integers(1, 6))
        msl = int(rng.choice([64, 130, 256]))
        lens = [int(x) for x in rng.integers(0, msl + 60, nb)]
        return Workload("rbj", B=nb, H=int(rng.integers(1, 3)), Dqk=dqk, Dv=dv, jagged=True, max_seq_len=msl,
                        max_len_draw=1, causal=causal), lens, False, None
    M = int(rng.integers(1, 400))
    N = M if causal else int(rng.integers(1, 400))
    w = Workload("rbd", B=int(rng.integers(1, 3)), H=int(rng.integers(1, 3)), M=M, N=N, Dqk=dqk, Dv=dv,
                 causal=causal)
    return w, None, rng.random() < 0.3, (int(rng.integers(0, 2)) if rng.random() < 0.3 else None)


@pytest.mark.parametrize("seed", list(range(16)))
def test_bwd_random_shapes(seed):
    """Seeded random draws (see _random_bwd_case): the library's forward
    then backward, every gradient against the float64 oracle."""
    rng = np.random.default_rng(500 + seed)
    w, lens, bias, mask_kind = _random_bwd_case(rng)
    f16 = rng.random() < 0.3
    inp = make_bwd_inputs(w, seed=600 + seed, lengths=lens)
    if w.jagged:
        cast = (lambda t: t.float().half()) if f16 else (lambda t: t)
        q, k, v, do = (cast(inp[n]).cuda() for n in ("q", "k", "v", "do"))
        kw = dict(causal=w.causal, sm_scale=inp["sm_scale"], offsets=inp["offsets"].cuda(),
                  max_seq_len=w.max_seq_len)
        o, lse = binding.attn_fwd(q, k, v, **kw)
        dq, dk, dv, delta = binding.attn_bwd(q, k, v, o, lse, do, **kw)
        assert binding.sync_check() == 0
        got = tuple(t.float().cpu().numpy() for t in (dq, dk, dv, delta))
        ref = oracle.attention_bwd_jagged(*(cast(inp[n]) for n in ("q", "k", "v", "do")), inp["offsets"],
                                          w.max_seq_len, causal=w.causal, sm_scale=inp["sm_scale"])
    else:
        g = torch.Generator().manual_seed(700 + seed)
        if bias:
            inp["bias"] = torch.randn((w.B, w.H, w.M, w.N), generator=g)
        if mask_kind == 0:
            m = torch.zeros((w.B, 1, 1, w.N), dtype=torch.uint8)
            for b in range(w.B):
                m[b, ..., : int(torch.randint(0, w.N + 1, (1,), generator=g))] = 1
            inp["mask"] = m
        elif mask_kind == 1:
            inp["mask"] = (torch.rand((w.B, w.H, w.M, w.N), generator=g) < 0.6).to(torch.uint8)
        got = run_gpu_bwd(inp, f16=f16)
        ref = oracle_bwd(inp, f16=f16)
    assert_grads_close(got, ref, what=f"seed {seed}: {w} bias={bias} mask={mask_kind} f16={f16}")
