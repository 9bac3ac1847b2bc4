#!/usr/bin/env python
"""Benchmark: attention forward + JVP TFLOP/s on one GB300 (per rank).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload causal|noncausal|jagged|bias_mask|tiny] [--op fwd_jvp|bwd]

A step is one fused forward + JVP pass (one launch of the library's kernel)
over the workload's synthetic inputs, already resident in HBM.  FLOPs are
algorithmic: 6 * (Dqk + Dv) per score element (three QK-shaped and three
PV-shaped matmuls), halved for causal attention.  Prints ONE JSON line on
rank 0.  Under torchrun every rank runs an independent replica of the
workload on its own GPU (no collective on the data path); the timed region
is bracketed by barriers and the slowest rank's time is used.

--impl reference times the float64 CPU oracle on the host cores (rank 0
only) on a bounded sample of the same workload: each step is one head.

--op fwd_f8 measures the FP8 (e5m2) forward (q, k, v in e5m2, V
transposed, O in e5m2) on a dense workload: a step is one launch; FLOPs are
the forward's two matmuls per score element; the roofline peak is the
measured bf16 peak times the nominal fp8 / bf16 rate (2).

--op bwd measures the attention backward instead (dense workloads): a step
is one backward -- the Delta launch, the dQ pass and the dK / dV pass --
given the forward's O and LSE (computed before the timed region).  FLOPs
are the standard five matmuls per score element (S, dP, dV, dQ, dK), halved
for causal attention; the kernels recompute S and dP in both passes, which
earns no credit.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from attention_forward_jvp_gb300.workloads import (WORKLOADS, flops_bwd, flops_fwd, flops_fwd_jvp,  # noqa: E402
                                                   make_bwd_inputs, make_f8_inputs, make_inputs,
                                                   min_hbm_bytes, min_hbm_bytes_bwd, score_elements)

METRIC = "attn fwd+JVP TFLOP/s (bf16, 1xGB300) and fraction of dense bf16 tensor peak"
METRIC_BWD = "attn backward (dQ, dK, dV) TFLOP/s (bf16, 1xGB300) and fraction of dense bf16 tensor peak"
METRIC_F8 = "attn FP8 (e5m2) forward TFLOP/s (1xGB300) and fraction of the fp8 tensor peak"
FP8_OVER_BF16 = 4.5 / 2.25  # nominal dense fp8 : bf16 tensor rate of a GB300
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 10**6  # GB300 L2


def strip_comments(src: str) -> str:
    """C / C++ / CUDA source without its comments, blank lines and trailing
    blanks.  One pass: string and character literals are copied as they
    are, `//` runs to the end of the line, `/* */` to its close."""
    out = []
    i, n = 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash(backward: bool = False) -> str:
    """Hash of the code a line's kernels are built from: the sources with
    comments and blank lines removed, so an edit of the comments keeps the
    hash (and the profiles recorded for it).  The forward kernels do not
    include the backward's files."""
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "attention_forward_jvp_gb300", "csrc", "*")))
    if not backward:
        files = [f for f in files if not os.path.basename(f).startswith("attn_bwd")]
    files += sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))
    for f in files:
        with open(f, encoding="utf-8") as fh:
            h.update(os.path.basename(f).encode())
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def describe(w) -> str:
    if w.jagged:
        return (f"{w.name}: {w.B} sequences, lengths U{{1..{w.max_len_draw}}}, H{w.H} "
                f"Dqk{w.Dqk} Dv{w.Dv}, packed [H,T,D], fwd+JVP")
    return (f"{w.name}: B{w.B} H{w.H} M{w.M} N{w.N} Dqk{w.Dqk} Dv{w.Dv} "
            f"{'causal' if w.causal else 'non-causal'}{' +bias+mask' if w.bias else ''} fwd+JVP")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def roofline(flops: float, nbytes: float, seconds: float, pk: dict, pk_kind: str) -> dict:
    """Roofline of one launch of the forward kernel.  The bound is whichever
    takes longer at the measured peaks: the tensor time (flops at the bf16
    peak) or the HBM time (algorithmic bytes at the copy bandwidth); achieved
    is that unit's algorithmic work over the measured launch time, and the
    other unit's figure is kept beside it."""
    tf_peak = float(pk.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    gb_peak = float(pk.get("hbm_gbs", FALLBACK_HBM_GBS))
    tflops = flops / seconds / 1e12
    gbs = nbytes / seconds / 1e9
    if nbytes / (gb_peak * 1e9) > flops / (tf_peak * 1e12):
        return {"bound": "hbm", "achieved": gbs, "peak": gb_peak, "unit": "GB/s", "frac": gbs / gb_peak,
                "peak_kind": f"{pk_kind} copy bandwidth", "algorithmic_bytes": nbytes,
                "tflops": tflops, "tflops_frac": tflops / tf_peak}
    return {"bound": "tensor", "achieved": tflops, "peak": tf_peak, "unit": "TFLOP/s", "frac": tflops / tf_peak,
            "peak_kind": f"{pk_kind} bf16 burst (kernel timed alone)", "algorithmic_bytes": nbytes,
            "hbm_gbs": gbs}


_SAMPLER_CHILD = r"""
import ctypes, sys, time
nv = ctypes.CDLL("libnvidia-ml.so.1")
if nv.nvmlInit_v2() != 0:
    sys.exit(0)
h = ctypes.c_void_p()
key, period = sys.argv[1], float(sys.argv[2])
ok = False
if key.startswith("GPU-"):
    ok = nv.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(h)) == 0
elif key.startswith("PCI:"):
    ok = nv.nvmlDeviceGetHandleByPciBusId_v2(key[4:].encode(), ctypes.byref(h)) == 0
if not ok:
    ok = nv.nvmlDeviceGetHandleByIndex_v2(int(sys.argv[3]), ctypes.byref(h)) == 0
if not ok:
    sys.exit(0)
fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or nv.nvmlDeviceGetCurrentClocksThrottleReasons
c, m, r = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
print("ready", flush=True)
while True:
    t = time.monotonic()
    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) == 0:
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m))
        fn(h, ctypes.byref(r))
        sys.stdout.write("%.6f %d %d %d\n" % (t, c.value, m.value, r.value))
        sys.stdout.flush()
    time.sleep(period)
"""


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons of one GPU
    every millisecond through NVML (read-only queries), in a child process
    of its own, so that the sampling takes no time from the thread that
    launches the timed kernels.  mark() records, on the system-wide
    monotonic clock, the instant from which samples belong to a region."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.001):
        self.period = period_s
        self.device_index = device_index
        self.marks = [("warmup", time.monotonic())]
        self.samples = []  # (time, sm_mhz, max_mhz, reasons)
        self.proc = None
        self.key = str(device_index)
        try:
            props = torch.cuda.get_device_properties(device_index)
            uid = getattr(props, "uuid", None)
            if uid is not None:
                self.key = str(uid) if str(uid).startswith("GPU-") else "GPU-" + str(uid)
            elif hasattr(props, "pci_bus_id"):
                self.key = "PCI:%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                                    getattr(props, "pci_device_id", 0))
        except Exception:
            pass

    def mark(self, tag):
        self.marks.append((tag, time.monotonic()))

    def __enter__(self):
        import subprocess
        try:
            self.proc = subprocess.Popen([sys.executable, "-c", _SAMPLER_CHILD, self.key, str(self.period),
                                          str(self.device_index)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            if self.proc.stdout.readline().strip() != "ready":
                self.proc.wait(timeout=5)
                self.proc = None
        except Exception:
            self.proc = None
        self.marks = [("warmup", time.monotonic())]
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            f = line.split()
            if len(f) == 4:
                self.samples.append((float(f[0]), int(f[1]), int(f[2]), int(f[3])))

    def _tag(self, t):
        tag = self.marks[0][0]
        for name, t0 in self.marks:
            if t >= t0:
                tag = name
        return tag

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "unavailable" if self.proc is None else "nvml"}
        timed = [s for s in self.samples if self._tag(s[0]) == "timed"]
        use = timed if timed else self.samples
        reasons = set()
        for _, _, _, r in use:
            for bit, nm in self.REASONS.items():
                if r & bit:
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(s[1] for s in use), "sm_max_mhz": max(s[2] for s in use),
                "reasons": sorted(reasons), "samples": len(use),
                "window": "timed region" if timed else "warm-up + timed region",
                "source": "nvml in a child process, every %d ms" % round(self.period * 1000)}


def dist_setup(impl):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and impl == "ours":
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


# ------------------------------------------------------------ CPU baseline
def oracle_sample(w, inp, n_units: int, start: int = 0):
    """Run the oracle on a bounded sample of the workload: ``n_units``
    heads (dense: whole (b, h) heads; jagged: (sequence, all heads)).
    Returns (seconds, algorithmic flops of the sample, description)."""
    import oracle
    if w.jagged:
        off = inp["offsets"].numpy()
        seqs = [(start + i) % w.B for i in range(n_units)]
        t0 = time.perf_counter()
        oracle.attention_fwd_jvp_jagged(inp["q"], inp["k"], inp["v"], inp["tq"], inp["tk"], inp["tv"],
                                        inp["offsets"], w.max_seq_len, causal=w.causal,
                                        sm_scale=inp["sm_scale"], only_seqs=set(seqs))
        dt = time.perf_counter() - t0
        lens = np.minimum(off[1:] - off[:-1], w.max_seq_len)[seqs].astype(np.float64)
        fl = 6.0 * (w.Dqk + w.Dv) * float((lens ** 2).sum()) * w.H * (0.5 if w.causal else 1.0)
        return dt, fl, oracle_sample_desc(w, n_units)
    BH = w.B * w.H
    units = [(start + i) % BH for i in range(n_units)]
    q64 = {n: None for n in ("q", "k", "v", "tq", "tk", "tv")}
    t0 = time.perf_counter()
    for u in units:
        b, h = divmod(u, w.H)
        for n in q64:
            q64[n] = oracle.to_f64(inp[n][b, h])
        bias = None if inp["bias"] is None else oracle.to_f64(inp["bias"][b, h])
        mask = None
        if inp["mask"] is not None:
            mk = inp["mask"]
            mask = np.broadcast_to(oracle.to_f64(mk[b if mk.shape[0] > 1 else 0, h if mk.shape[1] > 1 else 0]) != 0,
                                   (w.M, w.N))
        oracle.head_fwd_jvp(q64["q"], q64["k"], q64["v"], q64["tq"], q64["tk"], q64["tv"],
                            inp["sm_scale"], w.causal, bias, mask)
    dt = time.perf_counter() - t0
    fl = 6.0 * (w.Dqk + w.Dv) * w.M * w.N * n_units * (0.5 if w.causal else 1.0)
    return dt, fl, oracle_sample_desc(w, n_units)


def oracle_sample_desc(w, n_units: int) -> str:
    if w.jagged:
        return f"{n_units} sequences x {w.H} heads of the {w.name} workload"
    return (f"{n_units} of {w.B * w.H} (batch, head) pairs of the {w.name} workload, all rows, "
            "float64 NumPy (the oracle computes the full score matrix even when causal)")


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    inp = make_inputs(w, seed=0)
    for i in range(args.warmup):
        oracle_sample(w, inp, 1, start=i)
    times, flops = [], 0.0
    desc = ""
    for i in range(args.steps):
        dt, fl, desc = oracle_sample(w, inp, 1, start=args.warmup + i)
        times.append(dt)
        flops = fl
    tot = sum(times)
    value = flops * args.steps / tot / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": describe(w), "sample_per_step": "one head"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------- ours
def run_ours(args, w, world, rank, local):
    from attention_forward_jvp_gb300 import binding
    from attention_forward_jvp_gb300 import build as _b

    if not os.path.exists(_b.LIB_PATH):
        _b.build()
    binding.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = make_inputs(w, seed=0)
    d = {n: inp[n].to(dev) for n in ("q", "k", "v", "tq", "tk", "tv")}
    kw = dict(causal=w.causal, sm_scale=inp["sm_scale"],
              offsets=None if inp["offsets"] is None else inp["offsets"].to(dev),
              max_seq_len=inp["max_seq_len"],
              bias=None if inp["bias"] is None else inp["bias"].to(dev),
              mask=None if inp["mask"] is None else inp["mask"].to(dev))
    flops = flops_fwd_jvp(w, inp["offsets"])
    out = binding.attn_fwd_jvp(d["q"], d["k"], d["v"], d["tq"], d["tk"], d["tv"], **kw)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.attn_fwd_jvp(d["q"], d["k"], d["v"], d["tq"], d["tk"], d["tv"], out=out, **kw)

    # Inputs that fit in L2 would be re-read from L2 by every step: such
    # workloads write a buffer twice the size of L2 before each step and time
    # each step with its own pair of events (the flush is not timed).
    flush = min_hbm_bytes(w, inp) < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            step()
        st = binding.sync_check(stream)
        if st != 0:
            raise RuntimeError(f"device error during warm-up: {binding.status_string(st)}")
        barrier(world)
        torch.cuda.synchronize()
        n0 = binding.launch_count()
        clk.mark("timed")
        if flush:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for i in range(args.steps):
                flush_buf.fill_(float(i))
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                step()
            e1.record(stream)
        torch.cuda.synchronize()
        clk.mark("after")
        barrier(world)
        launches = binding.launch_count() - n0
    st = binding.sync_check(stream)
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {binding.status_string(st)}")
    if flush:
        ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    else:
        ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world)
    value = world * flops / (ms_max * 1e-3) / 1e12
    # (the step is exactly one launch of the fused kernel, so ms, its
    # per-step device time measured on its stream, is also the launch
    # duration the roofline below divides by)

    # end to end through the public API with pinned host buffers
    host = {n: inp[n].pin_memory() for n in ("q", "k", "v", "tq", "tk", "tv")}
    hkw = dict(kw)
    for key in ("offsets", "bias", "mask"):
        if inp[key] is not None:
            hkw[key] = inp[key].pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    h2d += sum(hkw[k].numel() * hkw[k].element_size() for k in ("offsets", "bias", "mask") if hkw[k] is not None)
    e2e_steps = max(1, min(args.steps, 10))
    hout = binding.attn_fwd_jvp(*[host[n] for n in ("q", "k", "v", "tq", "tk", "tv")], **hkw)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        hout = binding.attn_fwd_jvp(*[host[n] for n in ("q", "k", "v", "tq", "tk", "tv")], **hkw)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_s = max_over_ranks(e2e_s, world)
    e2e_val = world * flops / e2e_s / 1e12

    if rank != 0:
        return 0
    pk, pk_kind = peaks()
    peak = float(pk.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    traffic = None
    tf = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tf):
        with open(tf) as fh:
            rec = json.load(fh).get(w.name)
        if rec and rec.get("kernel_hash") == kernel_source_hash():
            traffic = rec.get("dram_bytes_per_launch")
    roof = roofline(flops, min_hbm_bytes(w, inp), ms * 1e-3, pk, pk_kind)
    roof["traffic"] = traffic
    cpu = None
    if world == 1 and not args.skip_cpu_baseline:
        # heads (jagged: sequences) one at a time until about cpu_seconds of
        # oracle work, or the whole workload, whichever comes first
        n_all = w.B if w.jagged else w.B * w.H
        dt = fl = 0.0
        n = 0
        while n < n_all and (n == 0 or dt < args.cpu_seconds):
            d1, f1, _ = oracle_sample(w, inp, 1, start=n)
            dt += d1
            fl += f1
            n += 1
        desc = oracle_sample_desc(w, n)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": desc, "seconds": dt}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": describe(w), "flops_per_step": flops,
                   "l2": ("L2 flushed before each step (%d MB written), steps timed one by one"
                          % (2 * L2_BYTES // 10**6) if flush else "inputs larger than L2, no flush"),
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": value / world / peak,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "kernel_hash": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- backward
def oracle_sample_bwd(w, inp, n_units: int, start: int = 0):
    """The backward oracle on ``n_units`` whole (b, h) heads.  Returns
    (seconds, algorithmic flops of the sample)."""
    import oracle
    BH = w.B * w.H
    t0 = time.perf_counter()
    for i in range(n_units):
        b, h = divmod((start + i) % BH, w.H)
        oracle.head_bwd(*(oracle.to_f64(inp[n][b, h]) for n in ("q", "k", "v", "do")), inp["sm_scale"],
                        causal=w.causal)
    dt = time.perf_counter() - t0
    return dt, flops_bwd(w) / BH * n_units


def run_reference_bwd(args, w, world, rank):
    if rank != 0:
        return 0
    inp = make_bwd_inputs(w, seed=0)
    for i in range(args.warmup):
        oracle_sample_bwd(w, inp, 1, start=i)
    tot = fl = 0.0
    for i in range(args.steps):
        dt, f1 = oracle_sample_bwd(w, inp, 1, start=args.warmup + i)
        tot += dt
        fl = f1
    value = fl * args.steps / tot / 1e12
    desc = (f"each step: one of {w.B * w.H} (batch, head) pairs of the {w.name} workload, float64 NumPy "
            "(the oracle forms the full score matrix even when causal)")
    line = {
        "impl": "reference", "metric": METRIC_BWD, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": describe(w).replace("fwd+JVP", "backward"),
                                        "sample_per_step": "one head"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours_bwd(args, w, world, rank, local):
    from attention_forward_jvp_gb300 import binding
    from attention_forward_jvp_gb300 import build as _b

    if w.bias or w.mask_keep is not None or w.Dqk != w.Dv:
        raise SystemExit(f"--op bwd runs workloads without bias / mask and Dqk == Dv ({w.name} is not)")
    if not os.path.exists(_b.LIB_PATH):
        _b.build()
    binding.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = make_bwd_inputs(w, seed=0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    kw = dict(causal=w.causal, sm_scale=inp["sm_scale"],
              offsets=None if inp["offsets"] is None else inp["offsets"].to(dev),
              max_seq_len=inp["max_seq_len"])
    o, lse = binding.attn_fwd(q, k, v, **kw)
    out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(lse))
    flops = flops_bwd(w, inp["offsets"])
    elem = score_elements(w, inp["offsets"]) * (0.5 if w.causal else 1.0)
    flops_dkdv = 4.0 * (w.Dqk + w.Dv) * elem   # S^T, dP^T, dV, dK
    stream = torch.cuda.current_stream(dev)
    stages = (binding.BWD_DELTA, binding.BWD_DQ, binding.BWD_DKDV)

    flush = min_hbm_bytes_bwd(w, q.numel() // w.Dqk if w.jagged else None) < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            binding.attn_bwd(q, k, v, o, lse, do, out=out, **kw)
        st = binding.sync_check(stream)
        if st != 0:
            raise RuntimeError(f"device error during warm-up: {binding.status_string(st)}")
        barrier(world)
        torch.cuda.synchronize()
        n0 = binding.launch_count()
        clk.mark("timed")
        for i in range(args.steps):
            if flush:
                flush_buf.fill_(float(i))
            ev[i][0].record(stream)
            for j, sg in enumerate(stages):
                binding.attn_bwd(q, k, v, o, lse, do, out=out, stages=sg, **kw)
                ev[i][j + 1].record(stream)
        torch.cuda.synchronize()
        clk.mark("after")
        barrier(world)
        launches = binding.launch_count() - n0
    st = binding.sync_check(stream)
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {binding.status_string(st)}")
    per = [sum(e[j].elapsed_time(e[j + 1]) for e in ev) / args.steps for j in range(3)]
    ms = sum(per)
    ms_max = max_over_ranks(ms, world)
    value = world * flops / (ms_max * 1e-3) / 1e12

    # end to end through the public API with pinned host buffers
    hin = [t.cpu().pin_memory() for t in (q, k, v, o, lse, do)]
    hkw = dict(kw)
    if inp["offsets"] is not None:
        hkw["offsets"] = inp["offsets"].pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hin)
    h2d += 0 if inp["offsets"] is None else inp["offsets"].numel() * 4
    e2e_steps = max(1, min(args.steps, 10))
    hout = binding.attn_bwd(*hin, **hkw)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        hout = binding.attn_bwd(*hin, **hkw)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world)
    e2e_val = world * flops / e2e_s / 1e12

    if rank != 0:
        return 0
    pk, pk_kind = peaks()
    peak = float(pk.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    achieved = flops_dkdv / (per[2] * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": None,
            "kernel": "dK/dV pass (attn_bwd_kernel<D, KV=true>): S^T, dP^T, dV, dK",
            "peak_kind": f"{pk_kind} bf16 burst (kernel timed alone)",
            "stage_ms": {"delta": per[0], "dq": per[1], "dkdv": per[2]},
            "stage_tflops": {"dq": 2.0 * (2 * w.Dqk + w.Dv) * elem / (per[1] * 1e-3) / 1e12,
                             "dkdv": achieved},
            "delta_gbs": 2.0 * 2 * (o.numel() // w.Dv) * w.Dv / (per[0] * 1e-3) / 1e9}
    cpu = None
    if world == 1 and not args.skip_cpu_baseline and not w.jagged:
        dt = fl = 0.0
        n = 0
        while n < w.B * w.H and (n == 0 or dt < args.cpu_seconds):
            d1, f1 = oracle_sample_bwd(w, inp, 1, start=n)
            dt += d1
            fl += f1
            n += 1
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"{n} of {w.B * w.H} (batch, head) pairs of the {w.name} workload, float64 NumPy",
               "seconds": dt}
    line = {
        "metric": METRIC_BWD, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": describe(w).replace("fwd+JVP", "backward"), "flops_per_step": flops,
                   "l2": ("L2 flushed before each step (%d MB written)" % (2 * L2_BYTES // 10**6)
                          if flush else "inputs larger than L2, no flush"),
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": value / world / peak,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "kernel_hash": kernel_source_hash(backward=True),
    }
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------- fp8 forward
def oracle_sample_f8(w, inp, n_units: int, start: int = 0):
    import oracle
    BH = w.B * w.H
    t0 = time.perf_counter()
    for i in range(n_units):
        b, h = divmod((start + i) % BH, w.H)
        oracle.head_fwd_e5m2(*(oracle.to_f64(inp[n][b, h]) for n in ("q", "k", "v")), inp["sm_scale"],
                             causal=w.causal)
    return time.perf_counter() - t0, flops_fwd(w) / BH * n_units


def run_reference_f8(args, w, world, rank):
    if rank != 0:
        return 0
    inp = make_f8_inputs(w, seed=0)
    for i in range(args.warmup):
        oracle_sample_f8(w, inp, 1, start=i)
    tot = fl = 0.0
    for i in range(args.steps):
        dt, fl = oracle_sample_f8(w, inp, 1, start=args.warmup + i)
        tot += dt
    value = fl * args.steps / tot / 1e12
    desc = f"each step: one of {w.B * w.H} (batch, head) pairs of the {w.name} workload in e5m2, float64 NumPy"
    line = {
        "impl": "reference", "metric": METRIC_F8, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w).replace("fwd+JVP", "FP8 forward"), "sample_per_step": "one head"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours_f8(args, w, world, rank, local):
    from attention_forward_jvp_gb300 import binding
    from attention_forward_jvp_gb300 import build as _b

    if w.jagged or w.bias or w.mask_keep is not None or w.Dqk != w.Dv or w.Dqk not in (64, 128):
        raise SystemExit(f"--op fwd_f8 runs dense workloads without bias / mask, D in {{64, 128}} ({w.name} is not)")
    if not os.path.exists(_b.LIB_PATH):
        _b.build()
    binding.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = make_f8_inputs(w, seed=0)
    q, k, vt = (inp[n].to(dev) for n in ("q", "k", "vt"))
    kw = dict(causal=w.causal, sm_scale=inp["sm_scale"])
    out = binding.attn_fwd_f8(q, k, vt, **kw)
    stream = torch.cuda.current_stream(dev)
    flops = flops_fwd(w)
    io_bytes = q.numel() + k.numel() + vt.numel() + out[0].numel() + out[1].numel() * 4
    flush = io_bytes < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            binding.attn_fwd_f8(q, k, vt, out=out, **kw)
        st = binding.sync_check(stream)
        if st != 0:
            raise RuntimeError(f"device error during warm-up: {binding.status_string(st)}")
        barrier(world)
        torch.cuda.synchronize()
        n0 = binding.launch_count()
        clk.mark("timed")
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            if flush:
                flush_buf.fill_(float(i))
            ev[i][0].record(stream)
            binding.attn_fwd_f8(q, k, vt, out=out, **kw)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        clk.mark("after")
        barrier(world)
        launches = binding.launch_count() - n0
    st = binding.sync_check(stream)
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {binding.status_string(st)}")
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    ms_max = max_over_ranks(ms, world)
    value = world * flops / (ms_max * 1e-3) / 1e12
    hin = [inp[n].pin_memory() for n in ("q", "k", "vt")]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    hout = binding.attn_fwd_f8(*hin, **kw)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    e2e_steps = max(1, min(args.steps, 10))
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        hout = binding.attn_fwd_f8(*hin, **kw)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world)
    if rank != 0:
        return 0
    pk, pk_kind = peaks()
    peak = float(pk.get("bf16_tflops", FALLBACK_BF16_TFLOPS)) * FP8_OVER_BF16
    achieved = flops / (ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": None, "kernel": "attn_fwd_kernel<D, D, no JVP, no bias, e5m2>",
            "peak_kind": f"{pk_kind} bf16 burst x {FP8_OVER_BF16:g} (nominal fp8 / bf16 dense rate)",
            "algorithmic_bytes": io_bytes, "hbm_gbs": io_bytes / (ms * 1e-3) / 1e9}
    cpu = None
    if world == 1 and not args.skip_cpu_baseline:
        dt = fl = 0.0
        n = 0
        while n < w.B * w.H and (n == 0 or dt < args.cpu_seconds):
            d1, f1 = oracle_sample_f8(w, inp, 1, start=n)
            dt += d1
            fl += f1
            n += 1
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"{n} of {w.B * w.H} (batch, head) pairs of the {w.name} workload in e5m2, float64 NumPy",
               "seconds": dt}
    line = {
        "metric": METRIC_F8, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e5m2", "data": "synthetic",
        "config": {"workload": describe(w).replace("fwd+JVP", "FP8 forward"), "flops_per_step": flops,
                   "l2": ("L2 flushed before each step (%d MB written)" % (2 * L2_BYTES // 10**6)
                          if flush else "inputs larger than L2, no flush"),
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": value / world / peak,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": world * flops / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "kernel_hash": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="causal", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="approximate seconds of oracle work in the CPU-baseline sample")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="fwd_jvp", choices=["fwd_jvp", "bwd", "fwd_f8"],
                    help="fwd_jvp: the fused forward + JVP (default); bwd: the backward; "
                         "fwd_f8: the FP8 (e5m2) forward")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = WORKLOADS[args.workload]
    world, rank, local = dist_setup(args.impl)
    if args.op == "bwd":
        rc = (run_reference_bwd(args, w, world, rank) if args.impl == "reference"
              else run_ours_bwd(args, w, world, rank, local))
    elif args.op == "fwd_f8":
        rc = (run_reference_f8(args, w, world, rank) if args.impl == "reference"
              else run_ours_f8(args, w, world, rank, local))
    elif args.impl == "reference":
        rc = run_reference(args, w, world, rank)
    else:
        rc = run_ours(args, w, world, rank, local)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
