"""The C-ABI library builds, loads and exports what include/attn_jvp.h
declares; argument validation returns its status codes without touching
a GPU (no compute call is made here)."""
import ctypes
import math
import os
import re

import pytest

from attention_forward_jvp_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(L):
    declared = _declared_functions()
    assert declared, "no declarations found"
    for name in declared:
        assert hasattr(L, name), f"{name} declared but not exported"
    assert declared == set(binding.EXPORTS)


def test_status_strings(L):
    for s in range(6):
        assert binding.status_string(s)
    assert binding.status_string(99) == "unknown status"


def _shape(B=1, H=1, M=128, N=128, Dqk=64, Dv=64, T=0, msl=0):
    s = binding.AttnShape()
    s.B, s.H, s.M, s.N, s.Dqk, s.Dv, s.T, s.max_seq_len = B, H, M, N, Dqk, Dv, T, msl
    return s


FAKE = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced (validation fails first)


def _call(L, shape, q=FAKE, k=FAKE, v=FAKE, tq=FAKE, tk=FAKE, tv=FAKE, offsets=None, bias=None,
          causal=0, scale=float("nan"), o=FAKE, to=FAKE, lse=FAKE):
    return L.attn_fwd_jvp(ctypes.byref(shape) if shape is not None else None, q, k, v, tq, tk, tv,
                          offsets, bias, causal, scale, o, to, lse, None)


def test_rejects_null_shape(L):
    assert _call(L, None) == 1


def test_rejects_unsupported_head_dims(L):
    # the forward takes Dqk, Dv in {16, 32, 64, 128, 256}, with and without
    # tangents; other widths are refused before anything is launched
    assert _call(L, _shape(Dqk=8)) == 2
    assert _call(L, _shape(Dqk=96)) == 2
    assert _call(L, _shape(Dv=48)) == 2
    assert _call(L, _shape(Dqk=512, Dv=64)) == 2
    assert _call(L, _shape(Dqk=64, Dv=320)) == 2


def test_rejects_causal_cross_attention(L):
    assert _call(L, _shape(M=128, N=256), causal=1) == 1


def test_rejects_negative_sizes_and_bad_scale(L):
    assert _call(L, _shape(M=-1)) == 1
    assert _call(L, _shape(B=-2)) == 1
    assert _call(L, _shape(), scale=-1.0) == 1
    assert _call(L, _shape(), scale=math.inf) == 1
    assert _call(L, _shape(), scale=0.0) == 1


def test_rejects_null_tangents(L):
    assert _call(L, _shape(), tq=None) == 1
    assert _call(L, _shape(), tk=None) == 1
    assert _call(L, _shape(), to=None) == 1
    assert _call(L, _shape(), lse=None) == 1


def test_rejects_misaligned(L):
    bad = ctypes.c_void_p(0x10008)
    assert _call(L, _shape(), q=bad) == 3
    assert _call(L, _shape(), tv=bad) == 3
    assert _call(L, _shape(), o=bad) == 3


def test_bias_with_jagged_is_unsupported(L):
    b = binding.AttnBias()
    b.bias = 0x10000
    off = ctypes.c_void_p(0x20000)
    assert _call(L, _shape(T=100, msl=64), offsets=off, bias=ctypes.byref(b)) == 2


def test_empty_problem_is_a_no_op(L):
    # nothing to compute: returns OK without touching any pointer or GPU
    assert _call(L, _shape(M=0), q=None, o=None, lse=None) == 0
    assert _call(L, _shape(B=0)) == 0
    assert L.attn_fwd(ctypes.byref(_shape(H=0)), None, None, None, None, None, 0,
                      float("nan"), None, None, None) == 0


def test_forward_only_validation(L):
    s = _shape(Dqk=128, Dv=24)
    assert L.attn_fwd(ctypes.byref(s), FAKE, FAKE, FAKE, None, None, 0, float("nan"), FAKE, FAKE, None) == 2


def test_timeout_setter_and_debug_hook_are_callable(L):
    L.attn_set_wait_timeout_ns(5)
    L.attn_set_wait_timeout_ns(2_000_000_000)
    L.attn_debug_skip_first_load(0)
    assert L.attn_launch_count() >= 0


def _bwd(L, shape, q=FAKE, k=FAKE, v=FAKE, o=FAKE, do=FAKE, lse=FAKE, offsets=None, bias=None,
         causal=0, scale=float("nan"), dq=FAKE, dk=FAKE, dv=FAKE, delta=FAKE, f16=False):
    fn = L.attn_bwd_f16 if f16 else L.attn_bwd
    return fn(ctypes.byref(shape) if shape is not None else None, q, k, v, o, do, lse, offsets,
              bias, causal, scale, dq, dk, dv, delta, None)


def test_bwd_validation(L):
    assert _bwd(L, None) == 1
    assert _bwd(L, _shape(Dqk=64, Dv=256)) == 2          # Dv outside {16, 32, 64, 128}
    assert _bwd(L, _shape(Dqk=256, Dv=256)) == 2
    assert _bwd(L, _shape(Dqk=8, Dv=8), f16=True) == 2
    off = ctypes.c_void_p(0x20000)
    assert _bwd(L, _shape(T=-1, msl=64), offsets=off) == 1          # jagged, bad T
    assert _bwd(L, _shape(T=100, msl=-2), offsets=off) == 1         # jagged, bad cap
    assert _bwd(L, _shape(T=100, msl=64, Dqk=96, Dv=64), offsets=off) == 2
    assert _bwd(L, _shape(T=0, msl=64), offsets=off) == 0           # no tokens: no-op
    b = binding.AttnBias()
    b.mask = 0x10000
    # a bias / mask with jagged inputs (dense only, as in the forward)
    assert _bwd(L, _shape(T=100, msl=64), offsets=off, bias=ctypes.byref(b)) == 2
    b.bias = 0x10002  # a bias not 4-byte aligned
    assert _bwd(L, _shape(), bias=ctypes.byref(b)) == 3
    assert _bwd(L, _shape(M=128, N=256), causal=1) == 1
    assert _bwd(L, _shape(), scale=-1.0) == 1
    assert _bwd(L, _shape(M=-3)) == 1
    assert _bwd(L, _shape(), lse=None) == 1
    assert _bwd(L, _shape(), dv=None) == 1
    assert _bwd(L, _shape(), delta=None) == 1
    bad = ctypes.c_void_p(0x10008)
    assert _bwd(L, _shape(), do=bad) == 3
    assert _bwd(L, _shape(), dk=bad) == 3
    # nothing to write: OK without touching a pointer or the GPU
    assert _bwd(L, _shape(B=0)) == 0
    assert _bwd(L, _shape(M=0, N=0), q=None, k=None, v=None) == 0


def test_bwd_stages_validation(L):
    def st(stages, shape=None):
        s = shape or _shape()
        return L.attn_bwd_stages(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 0,
                                 float("nan"), FAKE, FAKE, FAKE, FAKE, 0, stages, None)
    assert st(0) == 1            # no stage selected
    assert st(8) == 1            # unknown stage bit
    assert st(7, _shape(B=0)) == 0
    assert st(2, _shape(Dqk=256, Dv=128)) == 2


def test_plain_c_caller_compiles_links_and_validates(L, tmp_path):
    """tests/c/abi_from_c.c, a C99 program using only include/attn_jvp.h,
    compiles with -pedantic, links against the library and gets the
    documented status codes back from calls that need no GPU."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "abi_from_c")
    libdir = os.path.dirname(build.LIB_PATH)
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_from_c.c"), "-o", exe, "-L", libdir, "-l:libattn_jvp.so",
           "-Wl,-rpath," + libdir, "-Wl,--allow-shlib-undefined", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().splitlines()[-1] == "0", r.stdout + r.stderr
