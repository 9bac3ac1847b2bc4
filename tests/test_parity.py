"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (the target's, written here): O max abs error <= 1e-2,
tO max abs error <= 2e-2 * max(1, ||tO_oracle||_inf), LSE max abs error
<= 1e-3; -inf LSE (empty rows) must match exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_jvp_gb300 import binding, build
from attention_forward_jvp_gb300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
T_TOL = 2e-2
L_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.lib()


def dev(x):
    return None if x is None else x.cuda()


def run_gpu(inp, jvp=True, nan_prefill=False):
    """Run the library on the CPU-drawn inputs; returns float numpy (O, [tO,] LSE).
    ``nan_prefill``: the outputs start as NaN, so a row the launch never
    writes stays NaN and fails the comparison."""
    q, k, v, tq, tk, tv = (dev(inp[n]) for n in ("q", "k", "v", "tq", "tk", "tv"))
    kw = dict(causal=inp["causal"], sm_scale=inp["sm_scale"], offsets=dev(inp["offsets"]),
              max_seq_len=inp["max_seq_len"], bias=dev(inp["bias"]), mask=dev(inp["mask"]))
    out = None
    if nan_prefill:
        shp = tuple(q.shape[:-1]) + (v.shape[-1],)
        o = torch.full(shp, float("nan"), dtype=q.dtype, device=q.device)
        lse = torch.full(shp[:-1], float("nan"), dtype=torch.float32, device=q.device)
        out = (o, torch.full_like(o, float("nan")), lse) if jvp else (o, lse)
    if jvp:
        out = binding.attn_fwd_jvp(q, k, v, tq, tk, tv, out=out, **kw)
    else:
        out = binding.attn_fwd(q, k, v, out=out, **kw)
    assert binding.sync_check() == 0
    return tuple(o.float().cpu().numpy() for o in out)


def assert_close(O, tO, L, Or, tOr, Lr, what=""):
    assert np.isfinite(O).all() and np.isfinite(tO).all(), f"{what}: non-finite output"
    eo = np.abs(O - Or).max() if O.size else 0.0
    tscale = max(1.0, np.abs(tOr).max() if tOr.size else 0.0)
    et = np.abs(tO - tOr).max() if tO.size else 0.0
    inf_r = np.isneginf(Lr)
    assert np.array_equal(np.isneginf(L), inf_r), f"{what}: empty-row LSE pattern differs"
    el = np.abs(L[~inf_r] - Lr[~inf_r]).max() if (~inf_r).any() else 0.0
    assert eo <= O_TOL, f"{what}: O err {eo:.3e}"
    assert et <= T_TOL * tscale, f"{what}: tO err {et:.3e} (scale {tscale:.2f})"
    assert el <= L_TOL, f"{what}: LSE err {el:.3e}"
    return eo, et, el


def oracle_dense(inp):
    return oracle.attention_fwd_jvp(inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"],
                                    causal=inp["causal"], sm_scale=inp["sm_scale"],
                                    bias=inp["bias"], mask=inp["mask"])


# ------------------------------------------------------------ full configs
@pytest.mark.parametrize("name", ["tiny", "noncausal", "causal", "jagged", "bias_mask", "causal_d256"])
def test_full_size_whole_output(name):
    """Each benchmark workload at full size (the five configurations and
    the head-dim-256 line), in the launch configuration the benchmark times
    (persistent grid, snake unit order, jagged cost-ordered work list, head
    groups at Dqk = 256), into NaN-prefilled outputs; every element of O, tO
    and LSE against the float64 oracle over all heads (jagged: all
    sequences)."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    O, tO, L = run_gpu(inp, nan_prefill=True)
    assert not np.isnan(L).any(), f"{name}: {int(np.isnan(L).sum())} LSE entries never written"
    assert not np.isnan(O).any() and not np.isnan(tO).any(), f"{name}: output rows never written"
    if w.jagged:
        ref = oracle.attention_fwd_jvp_jagged(
            inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"], inp["offsets"],
            w.max_seq_len, causal=w.causal, sm_scale=inp["sm_scale"])
    else:
        ref = oracle_dense(inp)
    eo, et, el = assert_close(O, tO, L, *ref, what=name)
    print(f"{name}: O err {eo:.2e}, tO err {et:.2e}, LSE err {el:.2e}")


def test_full_size_forward_only_equals_jvp_primal():
    """attn_fwd at the causal workload's full size, NaN-prefilled: O and LSE
    bit-identical to the primal outputs of the forward + JVP launch."""
    inp = make_inputs(WORKLOADS["causal"])
    O, _, L = run_gpu(inp, nan_prefill=True)
    O2, L2 = run_gpu(inp, jvp=False, nan_prefill=True)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


@pytest.mark.parametrize("case", ["dense", "jagged"])
def test_many_units_per_cta_with_odd_tile_counts(case):
    """Units with odd key-tile counts, many per CTA: each unit boundary
    shifts which score buffer a unit's first tile uses, so the softmax
    warps' barrier phases must stay in order across boundaries.  Dense
    D = 64 with 15 key tiles per unit (8 x 16 x 8 = 1024 units); jagged
    D = 64 with 400 sequences of 64 k + 1 .. 64 k + 64 tokens (odd and
    even tile counts, one-tile units).  NaN-prefilled, whole output."""
    if case == "dense":
        w = Workload("odd", B=8, H=16, M=1024, N=960, Dqk=64, Dv=64, sm_scale=0.125)
        inp = make_inputs(w, seed=50)
        ref = None
    else:
        g = torch.Generator().manual_seed(51)
        lens = (64 * torch.randint(0, 7, (400,), generator=g) + torch.randint(1, 65, (400,), generator=g)).tolist()
        w = Workload("oddj", B=400, H=4, Dqk=64, Dv=64, jagged=True, max_seq_len=448, max_len_draw=1,
                     sm_scale=0.125)
        inp = make_inputs(w, seed=52, lengths=lens)
        ref = oracle.attention_fwd_jvp_jagged(inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"],
                                              inp["offsets"], 448, sm_scale=0.125)
    for rep in range(2):
        O, tO, L = run_gpu(inp, nan_prefill=True)
        assert not np.isnan(O).any() and not np.isnan(tO).any() and not np.isnan(L).any()
        if ref is None:
            ref = oracle_dense(inp)
        assert_close(O, tO, L, *ref, what=f"{case} run {rep}")


def test_inputs_written_by_the_kernels_just_before():
    """The forward kernel is launched as a programmatic dependent of the
    kernel before it on the stream, so its prologue may run while that
    kernel is still writing.  Here every input is produced on the device
    by kernels launched immediately before the call (no synchronisation),
    the last of them rewriting Q in place; the outputs start as NaN and
    every element is compared with the oracle."""
    B, H, N, D = 1, 6, 700, 64
    g = torch.Generator(device="cuda").manual_seed(81)
    dev_in = [torch.randn((B, H, N, D), generator=g, device="cuda", dtype=torch.float32) for _ in range(6)]
    q_src = dev_in[0].to(torch.bfloat16)
    inp = {"causal": True, "sm_scale": 0.125, "offsets": None, "max_seq_len": None, "bias": None, "mask": None}
    names = ("q", "k", "v", "tq", "tk", "tv")
    torch.cuda.synchronize()
    # launched back to back on the current stream, the attention call last
    bf = [t.to(torch.bfloat16) for t in dev_in]
    q = torch.zeros_like(q_src)
    q.copy_(q_src)
    o = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    to = torch.full_like(o, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    out = binding.attn_fwd_jvp(q, *bf[1:], causal=True, sm_scale=0.125, out=(o, to, lse))
    assert binding.sync_check() == 0
    for n, t in zip(names, [q] + bf[1:]):
        inp[n] = t.cpu()
    O, tO, L = (x.float().cpu().numpy() for x in out)
    assert_close(O, tO, L, *oracle_dense(inp), what="inputs written just before the call")


def _random_case(rng):
    """One seeded draw over the supported space: head dims for Q / K and V
    independently in {16, 32, 64, 128, 256}, dense (causal, cross-attention
    lengths, bias and / or key mask) or jagged (lengths around tile edges,
    causal or not), bf16 or fp16 storage."""
    dims = [16, 32, 64, 128, 256]
    dqk, dv = int(rng.choice(dims)), int(rng.choice(dims))
    jagged = rng.random() < 0.3
    causal = rng.random() < 0.4
    scale = float(rng.choice([0.125, 0.2, 1.0 / math.sqrt(dqk)]))
    if jagged:
        nb = int(rng.integers(1, 7))
        msl = int(rng.choice([64, 100, 200, 300]))
        lens = [int(x) for x in rng.integers(0, msl + 70, nb)]
        w = Workload("rj", B=nb, H=int(rng.integers(1, 4)), Dqk=dqk, Dv=dv, jagged=True, max_seq_len=msl,
                     max_len_draw=1, causal=causal, sm_scale=scale)
        return w, lens, None
    M = int(rng.integers(1, 520))
    N = M if causal else int(rng.integers(1, 520))
    bias = rng.random() < 0.35
    w = Workload("rd", B=int(rng.integers(1, 3)), H=int(rng.integers(1, 4)), M=M, N=N, Dqk=dqk, Dv=dv,
                 causal=causal, bias=bias, sm_scale=scale)
    mask_kind = int(rng.integers(0, 3)) if rng.random() < 0.35 else None
    return w, None, mask_kind


@pytest.mark.parametrize("seed", list(range(24)))
def test_random_shapes_whole_output(seed):
    """Seeded random draws over head dims, lengths, causal, bias / mask,
    jagged and fp16 (see _random_case); NaN-prefilled outputs, every
    element against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    w, lens, mask_kind = _random_case(rng)
    inp = make_inputs(w, seed=2000 + seed, lengths=lens)
    if mask_kind is not None:
        g = torch.Generator().manual_seed(3000 + seed)
        if mask_kind == 0:    # key padding per batch, [B, 1, 1, N]
            m = torch.zeros((w.B, 1, 1, w.N), dtype=torch.uint8)
            for b in range(w.B):
                m[b, ..., : int(torch.randint(0, w.N + 1, (1,), generator=g))] = 1
        elif mask_kind == 1:  # per (b, h) key mask with holes, [B, H, 1, N]
            m = (torch.rand((w.B, w.H, 1, w.N), generator=g) < 0.7).to(torch.uint8)
        else:                 # full [B, H, M, N] mask
            m = (torch.rand((w.B, w.H, w.M, w.N), generator=g) < 0.6).to(torch.uint8)
        inp["mask"] = m
    if rng.random() < 0.3:
        inp = _to_f16(inp)
    O, tO, L = run_gpu(inp, nan_prefill=True)
    assert not np.isnan(O).any() and not np.isnan(tO).any() and not np.isnan(L).any(), "unwritten output"
    if w.jagged:
        ref = oracle.attention_fwd_jvp_jagged(inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"],
                                              inp["offsets"], w.max_seq_len, causal=w.causal,
                                              sm_scale=inp["sm_scale"])
    else:
        ref = oracle_dense(inp)
    assert_close(O, tO, L, *ref, what=f"seed {seed}: {w}")


# ------------------------------------------------------------- edge shapes
EDGE = [
    # B, H, M, N, Dqk, Dv, causal
    (1, 2, 999, 999, 64, 64, True),
    (1, 2, 999, 999, 64, 64, False),
    (1, 2, 1024, 1024, 64, 64, True),
    (1, 2, 256, 1024, 64, 128, False),
    (1, 2, 1000, 15, 128, 64, False),
    (1, 2, 515, 999, 64, 64, False),
    (1, 2, 515, 999, 128, 128, False),
    (2, 3, 130, 70, 128, 64, False),
    (1, 1, 1, 1, 64, 64, True),
    (1, 2, 200, 1, 128, 128, False),
    (1, 1, 300, 300, 128, 128, True),
    (3, 2, 64, 200, 64, 128, False),
    # cross-attention shapes of the Triton fused-attention JVP tests
    # (M, N, Dqk, Dv), including head dims 16 and 32
    (1, 2, 1000, 15, 128, 32, False),
    (1, 2, 512, 512, 16, 32, False),
    (1, 2, 515, 999, 16, 32, False),
    (2, 3, 300, 300, 32, 32, True),
    (1, 2, 200, 260, 32, 128, False),
    (1, 2, 130, 70, 128, 16, False),
]


@pytest.mark.parametrize("B,H,M,N,Dqk,Dv,causal", EDGE)
def test_edge_shapes(B, H, M, N, Dqk, Dv, causal):
    w = Workload("edge", B=B, H=H, M=M, N=N, Dqk=Dqk, Dv=Dv, causal=causal,
                 input_std=0.5, tangent_std=0.5, sm_scale=0.5)
    inp = make_inputs(w, seed=20)
    assert_close(*run_gpu(inp), *oracle_dense(inp), what=str((B, H, M, N, Dqk, Dv, causal)))


def test_no_keys_gives_empty_rows():
    w = Workload("nokeys", B=1, H=2, M=130, N=0, Dqk=64, Dv=64)
    inp = make_inputs(w)
    O, tO, L = run_gpu(inp)
    assert np.all(O == 0) and np.all(tO == 0) and np.all(np.isneginf(L))


@pytest.mark.parametrize("causal", [False, True])
def test_jagged_edge_lengths(causal):
    lens = [1, 63, 64, 65, 127, 128, 129, 300, 0, 2, 255, 256, 257]
    w = Workload("jag", B=len(lens), H=3, Dqk=128, Dv=64, jagged=True, max_seq_len=200,
                 max_len_draw=1, causal=causal, sm_scale=0.125)
    inp = make_inputs(w, seed=3, lengths=lens)
    O, tO, L = run_gpu(inp)
    Or, tOr, Lr = oracle.attention_fwd_jvp_jagged(
        inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"], inp["offsets"], 200,
        causal=causal, sm_scale=0.125)
    assert_close(O, tO, L, Or, tOr, Lr, what=f"jagged causal={causal}")


def test_jagged_small_head_dims():
    lens = [1, 64, 65, 200, 0, 129]
    w = Workload("jag16", B=len(lens), H=2, Dqk=16, Dv=32, jagged=True, max_seq_len=160,
                 max_len_draw=1, sm_scale=0.25)
    inp = make_inputs(w, seed=21, lengths=lens)
    O, tO, L = run_gpu(inp)
    Or, tOr, Lr = oracle.attention_fwd_jvp_jagged(
        inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"], inp["offsets"], 160,
        sm_scale=0.25)
    assert_close(O, tO, L, Or, tOr, Lr, what="jagged Dqk16 Dv32")


def test_bias_and_mask_with_fully_masked_row():
    w = Workload("bm", B=2, H=3, M=150, N=333, Dqk=128, Dv=128, bias=True)
    inp = make_inputs(w, seed=4)
    g = torch.Generator().manual_seed(5)
    mask = (torch.rand((2, 3, 150, 333), generator=g) < 0.6).to(torch.uint8)
    mask[0, 1, 7, :] = 0      # a fully masked row
    mask[1, 2, 149, :] = 0
    inp["mask"] = mask
    O, tO, L = run_gpu(inp)
    Or, tOr, Lr = oracle_dense(inp)
    assert_close(O, tO, L, Or, tOr, Lr, what="bias+mask")
    assert np.isneginf(L[0, 1, 7]) and np.all(O[0, 1, 7] == 0) and np.all(tO[0, 1, 7] == 0)


def test_broadcast_bias_strides():
    w = Workload("bb", B=2, H=2, M=140, N=190, Dqk=64, Dv=64)
    inp = make_inputs(w, seed=6)
    g = torch.Generator().manual_seed(7)
    inp["bias"] = torch.randn((1, 2, 1, 190), generator=g)   # per-head key bias, broadcast
    inp["mask"] = (torch.arange(190) < 170).to(torch.uint8).view(1, 1, 1, 190)
    assert_close(*run_gpu(inp), *oracle_dense(inp), what="broadcast bias")


def test_bias_ring_shared_by_heads_causal():
    # bias [2, 1, 200, 200] shared by all heads, with causal attention: the
    # bias goes through a tensor map (rows 800 bytes apart) whose head
    # dimension has size 1
    w = Workload("bh", B=2, H=3, M=200, N=200, Dqk=128, Dv=128, causal=True)
    inp = make_inputs(w, seed=11)
    g = torch.Generator().manual_seed(12)
    inp["bias"] = torch.randn((2, 1, 200, 200), generator=g)
    assert_close(*run_gpu(inp), *oracle_dense(inp), what="bias shared by heads, causal")


def test_bias_ring_shared_by_batch_with_full_mask():
    # bias [1, 2, 260, 132] shared by the batch, with a full random mask
    # [3, 2, 260, 132]; ragged last query and key tiles
    w = Workload("bb2", B=3, H=2, M=260, N=132, Dqk=64, Dv=128)
    inp = make_inputs(w, seed=13)
    g = torch.Generator().manual_seed(14)
    inp["bias"] = torch.randn((1, 2, 260, 132), generator=g)
    inp["mask"] = (torch.rand((3, 2, 260, 132), generator=g) < 0.7).to(torch.uint8)
    assert_close(*run_gpu(inp), *oracle_dense(inp), what="bias shared by batch + mask")


@pytest.mark.parametrize("causal", [False, True])
def test_key_mask_with_dead_key_tiles(causal):
    # A mask that does not depend on the query row, [B, H, 1, N]: key tiles
    # with no kept key (one alone, runs of them, the ragged last tile) are
    # skipped by the softmax warps (P = H = 0, no exponentials).  Tiles with
    # a single kept key, nonzero mask values other than 1, and a different
    # pattern per (batch, head) around them.
    N = 64 * 40 + 17
    w = Workload("dk", B=2, H=2, M=N if causal else 130, N=N, Dqk=64, Dv=64, bias=True, causal=causal)
    inp = make_inputs(w, seed=41)
    g = torch.Generator().manual_seed(42)
    mask = (torch.rand((2, 2, 1, N), generator=g) < 0.8).to(torch.uint8) * 5
    for b in range(2):
        for h in range(2):
            dead = [3, 39, 40] + list(range(30 + b, 36 + h))
            for t in dead:
                mask[b, h, 0, 64 * t: 64 * t + 64] = 0
            mask[b, h, 0, 64 * 10: 64 * 11] = 0
            mask[b, h, 0, 64 * 10 + 17 * (b + 2 * h)] = 1   # a single kept key
    inp["mask"] = mask
    assert_close(*run_gpu(inp), *oracle_dense(inp), what=f"dead key tiles (causal={causal})")


@pytest.mark.parametrize("causal,bias", [(False, True), (True, True), (False, False)])
def test_key_mask_trims_the_key_range(causal, bias):
    """A key mask that does not depend on the query row ([B, H, 1, N]): a
    planning kernel finds each (b, h)'s last kept key and the units stop
    there.  Last kept key inside a tile and at a tile boundary, a (b, h)
    with no kept key at all (empty rows), a hole before the last key."""
    B, H, N = 3, 2, 64 * 9 + 13
    M = N if causal else 200
    w = Workload("kp", B=B, H=H, M=M, N=N, Dqk=128, Dv=64, bias=bias, causal=causal)
    inp = make_inputs(w, seed=61)
    mask = torch.ones((B, H, 1, N), dtype=torch.uint8)
    mask[0, :, :, 300:] = 0
    mask[1, 0] = 0
    mask[1, 1, :, 64 * 5:] = 0
    mask[2, :, :, 7] = 0
    inp["mask"] = mask
    O, tO, L = run_gpu(inp, nan_prefill=True)
    assert_close(O, tO, L, *oracle_dense(inp), what=f"trimmed keys causal={causal} bias={bias}")
    assert np.isneginf(L[1, 0]).all() and (O[1, 0] == 0).all() and (tO[1, 0] == 0).all()


def test_mask_without_bias():
    w = Workload("mo", B=2, H=2, M=190, N=300, Dqk=128, Dv=64)
    inp = make_inputs(w, seed=15)
    g = torch.Generator().manual_seed(16)
    inp["mask"] = (torch.rand((2, 1, 190, 300), generator=g) < 0.5).to(torch.uint8)
    assert_close(*run_gpu(inp), *oracle_dense(inp), what="mask only")


@pytest.mark.parametrize("Dv", [64, 128])
def test_outputs_16_byte_but_not_32_byte_aligned(Dv):
    # the epilogue uses 32-byte stores only when both outputs allow them
    w = Workload("al", B=1, H=2, M=200, N=130, Dqk=64, Dv=Dv)
    inp = make_inputs(w, seed=17)
    q, k, v, tq, tk, tv = (dev(inp[n]) for n in ("q", "k", "v", "tq", "tk", "tv"))
    n = w.B * w.H * w.M * Dv
    ob = torch.full((n + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    tb = torch.full((n + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = ob[8:].view(w.B, w.H, w.M, Dv)
    to = tb[8:].view(w.B, w.H, w.M, Dv)
    assert o.data_ptr() % 32 == 16 and to.data_ptr() % 32 == 16
    lse = torch.empty((w.B, w.H, w.M), dtype=torch.float32, device="cuda")
    binding.attn_fwd_jvp(q, k, v, tq, tk, tv, sm_scale=inp["sm_scale"], out=(o, to, lse))
    assert binding.sync_check() == 0
    assert torch.isnan(ob[:8].float()).all() and torch.isnan(tb[:8].float()).all()
    assert_close(o.float().cpu().numpy(), to.float().cpu().numpy(), lse.cpu().numpy(),
                 *oracle_dense(inp), what=f"16-byte aligned outputs Dv={Dv}")


# ----------------------------------------------------------- head dim 256
# Dqk and Dv each in {16, 32, 64, 128, 256}, as the pages' kernels accept
# them.  With tangents, Dv = 256 runs as two column slices of 128 (each its
# own work unit); Dqk = 256 keeps Q and tQ (128 KB) resident with one K
# stage, and reads a bias per thread.
D256_JVP = [
    ("256x256", dict(B=2, H=2, M=300, N=333, Dqk=256, Dv=256)),
    ("256x256_causal", dict(B=1, H=3, M=400, N=400, Dqk=256, Dv=256, causal=True)),
    ("256x256_bias_mask", dict(B=2, H=2, M=200, N=260, Dqk=256, Dv=256, bias=True, mask_keep=200)),
    ("256x64", dict(B=2, H=2, M=260, N=300, Dqk=256, Dv=64)),
    ("256x128_causal", dict(B=1, H=2, M=333, N=333, Dqk=256, Dv=128, causal=True)),
    ("256x32_bias", dict(B=1, H=2, M=200, N=150, Dqk=256, Dv=32, bias=True)),
    ("64x256", dict(B=2, H=2, M=200, N=333, Dqk=64, Dv=256)),
    ("128x256_causal", dict(B=1, H=2, M=300, N=300, Dqk=128, Dv=256, causal=True)),
    ("16x256_bias_mask", dict(B=1, H=2, M=130, N=200, Dqk=16, Dv=256, bias=True, mask_keep=150)),
    ("128x256_many_units", dict(B=2, H=8, M=1024, N=1024, Dqk=128, Dv=256, causal=True)),
    # eight (b, h): the causal Dqk = 256 units walk the heads in four groups
    ("256x256_causal_head_groups", dict(B=2, H=4, M=333, N=333, Dqk=256, Dv=256, causal=True)),
]


@pytest.mark.parametrize("name,kw", D256_JVP, ids=[c[0] for c in D256_JVP])
def test_head_dim_256_jvp(name, kw):
    inp = make_inputs(Workload("d256", input_std=0.5, tangent_std=0.5, **kw), seed=41)
    assert_close(*run_gpu(inp, nan_prefill=True), *oracle_dense(inp), what=f"JVP {name}")


D256_FWD = [
    ("256x256", dict(B=2, H=2, M=300, N=333, Dqk=256, Dv=256)),
    ("256x256_causal", dict(B=1, H=3, M=400, N=400, Dqk=256, Dv=256, causal=True)),
    ("256x256_bias_mask", dict(B=2, H=2, M=200, N=260, Dqk=256, Dv=256, bias=True, mask_keep=200)),
    ("256x64_bias", dict(B=2, H=2, M=260, N=300, Dqk=256, Dv=64, bias=True)),
    ("256x128", dict(B=1, H=2, M=333, N=200, Dqk=256, Dv=128)),
    ("64x256_causal", dict(B=1, H=2, M=300, N=300, Dqk=64, Dv=256, causal=True)),
    ("128x256_bias_mask", dict(B=2, H=2, M=150, N=270, Dqk=128, Dv=256, bias=True, mask_keep=180)),
]


@pytest.mark.parametrize("name,kw", D256_FWD, ids=[c[0] for c in D256_FWD])
def test_head_dim_256_forward(name, kw):
    inp = make_inputs(Workload("d256", input_std=0.5, **kw), seed=41)
    O, L = run_gpu(inp, jvp=False, nan_prefill=True)
    Or, _, Lr = oracle_dense(inp)
    assert_close(O, np.zeros_like(O), L, Or, np.zeros_like(Or), Lr, what=f"D256 {name}")


def test_head_dim_256_fp16():
    inp = make_inputs(Workload("d256h", B=1, H=2, M=260, N=300, Dqk=256, Dv=256, input_std=0.5,
                               tangent_std=0.5), seed=42)
    for n in ("q", "k", "v", "tq", "tk", "tv"):
        inp[n] = inp[n].to(torch.float16)
    Or, tOr, Lr = oracle_dense(inp)
    assert_close(*run_gpu(inp, nan_prefill=True), Or, tOr, Lr, what="D256 fp16 JVP")
    O, L = run_gpu(inp, jvp=False, nan_prefill=True)
    assert_close(O, np.zeros_like(O), L, Or, np.zeros_like(Or), Lr, what="D256 fp16 forward")


@pytest.mark.parametrize("Dqk,Dv", [(256, 256), (64, 256), (256, 64)])
def test_head_dim_256_jagged(Dqk, Dv):
    lens = [1, 63, 64, 65, 200, 0, 129, 300]
    w = Workload("j256", B=len(lens), H=2, Dqk=Dqk, Dv=Dv, jagged=True, max_seq_len=260,
                 max_len_draw=1, input_std=0.5, tangent_std=0.5, sm_scale=0.1)
    inp = make_inputs(w, seed=43, lengths=lens)
    O, tO, L = run_gpu(inp, nan_prefill=True)
    Or, tOr, Lr = oracle.attention_fwd_jvp_jagged(
        inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"], inp["offsets"], 260,
        sm_scale=0.1)
    assert_close(O, tO, L, Or, tOr, Lr, what=f"jagged {Dqk}x{Dv}")


# ------------------------------------------------------------- fp16 storage
def _to_f16(inp):
    """The same draws rounded to fp16; the oracle reads these fp16 values."""
    out = dict(inp)
    for n in ("q", "k", "v", "tq", "tk", "tv"):
        out[n] = inp[n].to(torch.float16)
    return out


@pytest.mark.parametrize("name,kw", [
    ("dense", dict(B=2, H=3, M=300, N=260, Dqk=128, Dv=64)),
    ("causal", dict(B=1, H=2, M=640, N=640, Dqk=128, Dv=128, causal=True)),
    ("d64", dict(B=2, H=2, M=400, N=700, Dqk=64, Dv=64)),
    ("bias", dict(B=2, H=2, M=256, N=512, Dqk=128, Dv=64, bias=True, mask_keep=400)),
    ("small", dict(B=1, H=2, M=515, N=999, Dqk=16, Dv=32)),
])
def test_fp16_storage(name, kw):
    inp = _to_f16(make_inputs(Workload("f16", **kw), seed=31))
    O, tO, L = run_gpu(inp)
    assert_close(O, tO, L, *oracle_dense(inp), what=f"fp16 {name}")


@pytest.mark.parametrize("f16", [False, True])
def test_whole_key_tiles_dense_noncausal(f16):
    """Dense non-causal problems with head dims <= 64, no bias or mask and N
    a multiple of 64 run a lean instantiation of the ping-pong kernel (no
    masking, jagged or causal decode): forward + JVP against the oracle,
    NaN-prefilled, with a query tail and small head dims; the forward only
    bit-identical to its primal outputs."""
    for kw, seed in ((dict(B=2, H=3, M=200, N=320, Dqk=64, Dv=64), 81),
                     (dict(B=1, H=2, M=130, N=64, Dqk=32, Dv=16), 82)):
        inp = make_inputs(Workload("lean", sm_scale=0.125, **kw), seed=seed)
        if f16:
            inp = _to_f16(inp)
        O, tO, L = run_gpu(inp, nan_prefill=True)
        assert_close(O, tO, L, *oracle_dense(inp), what=f"lean {kw} f16={f16}")
        O2, L2 = run_gpu(inp, jvp=False, nan_prefill=True)
        assert np.array_equal(O, O2) and np.array_equal(L, L2)


def test_fp16_jagged_and_forward_only():
    lens = [3, 64, 130, 257, 1]
    w = Workload("jf16", B=len(lens), H=2, Dqk=64, Dv=64, jagged=True, max_seq_len=300,
                 max_len_draw=1, sm_scale=0.125)
    inp = _to_f16(make_inputs(w, seed=32, lengths=lens))
    O, tO, L = run_gpu(inp)
    Or, tOr, Lr = oracle.attention_fwd_jvp_jagged(
        inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"], inp["offsets"], 300,
        sm_scale=0.125)
    assert_close(O, tO, L, Or, tOr, Lr, what="fp16 jagged")
    O2, L2 = run_gpu(inp, jvp=False)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


# -------------------------------------------------------- kernel invariants
@pytest.mark.parametrize("name", ["tiny", "edge_causal", "edge_bias"])
def test_forward_only_matches_jvp_primal_bitwise(name):
    if name == "tiny":
        inp = make_inputs(WORKLOADS["tiny"])
    elif name == "edge_causal":
        inp = make_inputs(Workload("e", B=1, H=2, M=777, N=777, Dqk=128, Dv=128, causal=True), seed=8)
    else:
        inp = make_inputs(Workload("e", B=1, H=2, M=300, N=500, Dqk=128, Dv=64, bias=True,
                                   mask_keep=420), seed=9)
    O, _, L = run_gpu(inp, jvp=True)
    O2, L2 = run_gpu(inp, jvp=False)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


def test_causal_rows_ignore_future_keys_bitwise():
    inp = make_inputs(Workload("c", B=1, H=2, M=640, N=640, Dqk=64, Dv=64, causal=True), seed=10)
    O, tO, L = run_gpu(inp)
    for nm in ("k", "v", "tk", "tv"):
        inp[nm] = inp[nm].clone()
        inp[nm][:, :, 400:] = 7.0
    O2, tO2, L2 = run_gpu(inp)
    assert np.array_equal(O[:, :, :400], O2[:, :, :400])
    assert np.array_equal(tO[:, :, :400], tO2[:, :, :400])
    assert np.array_equal(L[:, :, :400], L2[:, :, :400])


def test_guard_bands_and_nan_prefill():
    inp = make_inputs(Workload("g", B=1, H=2, M=333, N=200, Dqk=64, Dv=128), seed=11)
    guard = 4096
    n_o = 1 * 2 * 333 * 128
    n_l = 1 * 2 * 333
    ob = torch.full((n_o + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    tb = torch.full((n_o + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lb = torch.full((n_l + 2 * guard,), float("nan"), dtype=torch.float32, device="cuda")
    o = ob[guard:guard + n_o].view(1, 2, 333, 128)
    to = tb[guard:guard + n_o].view(1, 2, 333, 128)
    lse = lb[guard:guard + n_l].view(1, 2, 333)
    q, k, v, tq, tk, tv = (dev(inp[n]) for n in ("q", "k", "v", "tq", "tk", "tv"))
    binding.attn_fwd_jvp(q, k, v, tq, tk, tv, sm_scale=inp["sm_scale"], out=(o, to, lse))
    assert binding.sync_check() == 0
    for buf, n in ((ob, n_o), (tb, n_o), (lb, n_l)):
        assert torch.isnan(buf[:guard].float()).all() and torch.isnan(buf[guard + n:].float()).all()
        assert torch.isfinite(buf[guard:guard + n].float()).all()
    Or, tOr, Lr = oracle_dense(inp)
    assert_close(o.float().cpu().numpy(), to.float().cpu().numpy(), lse.cpu().numpy(), Or, tOr, Lr)


def test_host_buffers_end_to_end_match_device_path():
    inp = make_inputs(WORKLOADS["tiny"])
    O, tO, L = run_gpu(inp)
    ho, hto, hl = binding.attn_fwd_jvp(inp["q"].pin_memory(), inp["k"].pin_memory(),
                                       inp["v"].pin_memory(), inp["tq"].pin_memory(),
                                       inp["tk"].pin_memory(), inp["tv"].pin_memory(),
                                       sm_scale=inp["sm_scale"])
    assert ho.device.type == "cpu"
    assert np.array_equal(ho.float().numpy(), O) and np.array_equal(hto.float().numpy(), tO)
    assert np.array_equal(hl.numpy(), L)


@pytest.mark.parametrize("jvp", [True, False])
def test_chunked_host_path_matches_device_path_bitwise(jvp):
    # 2 x 8 (batch, head) slabs: the host path cuts them into chunks, each
    # on a stream of its own; each slab is an independent problem, so the
    # results are bit-identical to one call over the whole batch on the
    # device
    w = Workload("hc", B=2, H=8, M=200, N=200, Dqk=64, Dv=64, causal=True)
    inp = make_inputs(w, seed=21)
    assert binding._slab_chunks(binding.attn_fwd_jvp if jvp else binding.attn_fwd,
                                (inp["q"], inp["k"], inp["v"]), {}) == 2
    dev_out = run_gpu(inp, jvp=jvp)
    names = ("q", "k", "v", "tq", "tk", "tv") if jvp else ("q", "k", "v")
    fn = binding.attn_fwd_jvp if jvp else binding.attn_fwd
    host_out = fn(*[inp[n].pin_memory() for n in names], causal=True, sm_scale=inp["sm_scale"])
    assert all(t.device.type == "cpu" for t in host_out)
    for h, d in zip(host_out, dev_out):
        assert np.array_equal(h.float().numpy(), d)


def test_default_scale_is_inverse_sqrt_dqk():
    inp = make_inputs(Workload("s", B=1, H=1, M=128, N=128, Dqk=128, Dv=64), seed=12)
    inp["sm_scale"] = None
    O, tO, L = run_gpu(inp)
    inp2 = dict(inp, sm_scale=1.0 / math.sqrt(128))
    assert_close(O, tO, L, *oracle_dense(inp2), what="default scale")


# ----------------------------------------------------- failure detection
@pytest.mark.parametrize("shape", ["tiny", "d256"])
def test_timed_out_wait_is_reported_and_context_survives(shape):
    # d256: head dim 256 with tangents, whose K copies use chunk stages
    if shape == "tiny":
        inp = make_inputs(WORKLOADS["tiny"])
    else:
        inp = make_inputs(Workload("t256", B=1, H=2, M=300, N=400, Dqk=256, Dv=256, input_std=0.5,
                                   tangent_std=0.5), seed=44)
    q, k, v, tq, tk, tv = (dev(inp[n]) for n in ("q", "k", "v", "tq", "tk", "tv"))
    binding.set_wait_timeout_ns(100_000_000)
    binding.debug_skip_first_load(True)
    try:
        binding.attn_fwd_jvp(q, k, v, tq, tk, tv, sm_scale=inp["sm_scale"])
        st = binding.sync_check()
    finally:
        binding.debug_skip_first_load(False)
        binding.set_wait_timeout_ns(2_000_000_000)
    assert st == 5  # ATTN_ERR_TIMEOUT
    assert binding.sync_check() == 0  # cleared
    O, tO, L = run_gpu(inp)
    assert_close(O, tO, L, *oracle_dense(inp), what="after timeout")


@pytest.mark.parametrize("causal", [False, True])
def test_jagged_work_list_writes_every_row(causal):
    """The jagged launch walks a device-built, cost-ordered work list: with
    NaN-prefilled outputs every row of every sequence must be written."""
    lens = [700, 3, 129, 0, 512, 64, 65, 1000, 257, 31]
    w = Workload("jl", B=len(lens), H=4, Dqk=64, Dv=64, jagged=True, max_seq_len=900,
                 max_len_draw=1, causal=causal, sm_scale=0.125)
    inp = make_inputs(w, seed=13, lengths=lens)
    T = inp["q"].shape[1]
    d = {n: inp[n].cuda() for n in ("q", "k", "v", "tq", "tk", "tv")}
    o = torch.full((4, T, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    to = torch.full((4, T, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((4, T), float("nan"), dtype=torch.float32, device="cuda")
    binding.attn_fwd_jvp(d["q"], d["k"], d["v"], d["tq"], d["tk"], d["tv"], causal=causal,
                         sm_scale=0.125, offsets=inp["offsets"].cuda(), max_seq_len=900,
                         out=(o, to, lse))
    assert binding.sync_check() == 0
    O, tO, L = (x.float().cpu().numpy() for x in (o, to, lse))
    assert not np.isnan(O).any() and not np.isnan(tO).any() and not np.isnan(L).any()
    Or, tOr, Lr = oracle.attention_fwd_jvp_jagged(
        inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"], inp["offsets"], 900,
        causal=causal, sm_scale=0.125)
    assert_close(O, tO, L, Or, tOr, Lr, what=f"jagged list causal={causal}")
