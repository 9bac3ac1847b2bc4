"""Host logic of bench.py that needs no GPU: the kernel source hash that
keys the recorded DRAM traffic (profiles/traffic.json) to the code it was
measured on."""
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_strip_comments_keeps_code_and_literals():
    src = ("int a = 1; // line comment /* not a block\n"
           "/* block\n   // inside */ int b = 2;\n"
           "\n"
           "const char* s = \"a // b /* c */\";   \n"
           "char q = '\\'';  // a quote\n")
    out = bench.strip_comments(src)
    assert out.splitlines() == ["int a = 1;", "  int b = 2;",
                                "const char* s = \"a // b /* c */\";", "char q = '\\'';"]


def _copy_sources(dst):
    for sub in (os.path.join("attention_forward_jvp_gb300", "csrc"), "include"):
        shutil.copytree(os.path.join(ROOT, sub), os.path.join(dst, sub))


def test_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base_f, base_b = bench.kernel_source_hash(), bench.kernel_source_hash(backward=True)
    k = tmp_path / "attention_forward_jvp_gb300" / "csrc" / "attn_kernel.cuh"
    text = k.read_text()
    # a comment edit and blank lines: same hashes
    k.write_text("// an added comment line\n\n" + text.replace("namespace attn {", "namespace attn {  /* x */", 1))
    assert bench.kernel_source_hash() == base_f
    assert bench.kernel_source_hash(backward=True) == base_b
    # a code edit: both change (the backward includes the forward header)
    k.write_text(text.replace("namespace attn {", "namespace attn {\nconstexpr int kProbe = 1;", 1))
    assert bench.kernel_source_hash() != base_f
    assert bench.kernel_source_hash(backward=True) != base_b


def test_backward_sources_do_not_change_the_forward_hash(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base_f, base_b = bench.kernel_source_hash(), bench.kernel_source_hash(backward=True)
    b = tmp_path / "attention_forward_jvp_gb300" / "csrc" / "attn_bwd_kernel.cuh"
    b.write_text(b.read_text() + "\nconstexpr int kProbe = 2;\n")
    assert bench.kernel_source_hash() == base_f
    assert bench.kernel_source_hash(backward=True) != base_b


def test_host_path_chunking_decision():
    """Which host calls the binding cuts into (batch, head) slab chunks: a
    dense forward without bias, mask or offsets, contiguous, at least 8
    slabs and M a multiple of 4 (lse rows of a chunk stay 16-byte aligned);
    four chunks from 128 MB of inputs, else two."""
    import torch
    from attention_forward_jvp_gb300 import binding
    t = torch.zeros(2, 8, 200, 64, dtype=torch.bfloat16)
    six, three = (t,) * 6, (t,) * 3
    assert binding._slab_chunks(binding.attn_fwd_jvp, six, {}) == 2
    assert binding._slab_chunks(binding.attn_fwd, three, {"bias": None, "mask": None}) == 2
    big = torch.empty(2, 16, 4096, 128, dtype=torch.bfloat16)   # 32 MB each, 192 MB for six
    assert binding._slab_chunks(binding.attn_fwd_jvp, (big,) * 6, {}) == 4
    assert binding._slab_chunks(binding.attn_fwd, three, {"bias": t}) == 1
    assert binding._slab_chunks(binding.attn_fwd, three, {"mask": t}) == 1
    assert binding._slab_chunks(binding.attn_fwd, three, {"offsets": t}) == 1
    assert binding._slab_chunks(binding.attn_bwd, six, {}) == 1
    small = torch.zeros(1, 4, 200, 64, dtype=torch.bfloat16)
    assert binding._slab_chunks(binding.attn_fwd, (small,) * 3, {}) == 1      # 4 slabs
    odd = torch.zeros(2, 8, 202, 64, dtype=torch.bfloat16)
    assert binding._slab_chunks(binding.attn_fwd, (odd, t, t), {}) == 1       # M % 4 != 0
    strided = torch.zeros(2, 8, 64, 200, dtype=torch.bfloat16).transpose(2, 3)
    assert binding._slab_chunks(binding.attn_fwd, (strided, t, t), {}) == 1   # not contiguous
    jag = torch.zeros(8, 1000, 64, dtype=torch.bfloat16)
    assert binding._slab_chunks(binding.attn_fwd, (jag,) * 3, {}) == 1        # [H, T, D]


def test_roofline_bound_follows_the_longer_time():
    """bias + mask (77.3 GFLOP, 318.9 MB) is HBM-bound at the measured
    peaks (47.6 us of copies against 41.4 us of tensor work); the causal
    workload (412 GFLOP, 269 MB) is tensor-bound."""
    pk = {"bf16_tflops": 1868.7, "hbm_gbs": 6695.5}
    r = bench.roofline(77.3e9, 318.9e6, 107.4e-6, pk, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 318.9e6 / 107.4e-6 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 6695.5) < 1e-12
    assert abs(r["tflops"] - 77.3e9 / 107.4e-6 / 1e12) < 1e-9
    r = bench.roofline(412.3e9, 269.0e6, 276.1e-6, pk, "measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - 412.3e9 / 276.1e-6 / 1e12 / 1868.7) < 1e-12
