"""ctypes binding of the C ABI in include/attn_jvp.h.

Argument marshalling only: shapes, strides and raw pointers of torch
tensors are handed to ``libattn_jvp.so``; every arithmetic step runs in its
CUDA kernels.  Outputs are allocated with torch (device memory plumbing).
CPU (host) inputs are staged through the device: the host->device copies,
the kernel and the device->host copies all run on the current stream.

There is no fallback: if the library is missing or the GPU is absent the
call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

EXPORTS = (
    "attn_fwd_jvp",
    "attn_fwd",
    "attn_fwd_jvp_f16",
    "attn_fwd_f16",
    "attn_fwd_f8",
    "attn_fwd_jvp_noalloc",
    "attn_bwd",
    "attn_bwd_f16",
    "attn_bwd_stages",
    "attn_sync_check",
    "attn_status_string",
    "attn_launch_count",
    "attn_set_wait_timeout_ns",
    "attn_debug_skip_first_load",
)

STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
          3: "ATTN_ERR_MISALIGNED", 4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_TIMEOUT"}


class AttnShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("M", ctypes.c_int32),
                ("N", ctypes.c_int32), ("Dqk", ctypes.c_int32), ("Dv", ctypes.c_int32),
                ("T", ctypes.c_int64), ("max_seq_len", ctypes.c_int32)]


class AttnBias(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("bias_stride", ctypes.c_int64 * 4),
                ("mask", ctypes.c_void_p), ("mask_stride", ctypes.c_int64 * 4)]


class AttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


_LIB = None


def lib() -> ctypes.CDLL:
    """Open the library (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with attention_forward_jvp_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.attn_fwd_jvp.restype = i32
    L.attn_fwd_jvp.argtypes = [ctypes.POINTER(AttnShape), vp, vp, vp, vp, vp, vp, vp,
                               ctypes.POINTER(AttnBias), i32, f32, vp, vp, vp, vp]
    L.attn_fwd_jvp_noalloc.restype = i32
    L.attn_fwd_jvp_noalloc.argtypes = L.attn_fwd_jvp.argtypes
    L.attn_fwd_jvp_f16.restype = i32
    L.attn_fwd_jvp_f16.argtypes = L.attn_fwd_jvp.argtypes
    L.attn_fwd.restype = i32
    L.attn_fwd.argtypes = [ctypes.POINTER(AttnShape), vp, vp, vp, vp,
                           ctypes.POINTER(AttnBias), i32, f32, vp, vp, vp]
    L.attn_fwd_f16.restype = i32
    L.attn_fwd_f16.argtypes = L.attn_fwd.argtypes
    L.attn_bwd.restype = i32
    L.attn_bwd.argtypes = [ctypes.POINTER(AttnShape), vp, vp, vp, vp, vp, vp, vp,
                           ctypes.POINTER(AttnBias), i32, f32, vp, vp, vp, vp, vp]
    L.attn_bwd_f16.restype = i32
    L.attn_bwd_f16.argtypes = L.attn_bwd.argtypes
    L.attn_bwd_stages.restype = i32
    L.attn_bwd_stages.argtypes = [ctypes.POINTER(AttnShape), vp, vp, vp, vp, vp, vp, vp,
                                  ctypes.POINTER(AttnBias), i32, f32, vp, vp, vp, vp, i32,
                                  ctypes.c_uint, vp]
    L.attn_fwd_f8.restype = i32
    L.attn_fwd_f8.argtypes = [ctypes.POINTER(AttnShape), vp, vp, vp, i32, f32, vp, vp, vp]
    L.attn_sync_check.restype = i32
    L.attn_sync_check.argtypes = [vp]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_status_string.argtypes = [i32]
    L.attn_launch_count.restype = ctypes.c_uint64
    L.attn_launch_count.argtypes = []
    L.attn_set_wait_timeout_ns.restype = None
    L.attn_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    L.attn_debug_skip_first_load.restype = None
    L.attn_debug_skip_first_load.argtypes = [i32]
    _LIB = L
    return L


def _check(status: int):
    if status != 0:
        raise AttnError(status, lib().attn_status_string(status).decode())


def status_string(status: int) -> str:
    return lib().attn_status_string(status).decode()


def launch_count() -> int:
    return int(lib().attn_launch_count())


def sync_check(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise and return the device error status (0 = ok)."""
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(lib().attn_sync_check(ctypes.c_void_p(s.cuda_stream)))


def set_wait_timeout_ns(ns: int):
    lib().attn_set_wait_timeout_ns(int(ns))


def debug_skip_first_load(enable: bool):
    lib().attn_debug_skip_first_load(1 if enable else 0)


def _elem_type(q: torch.Tensor):
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"inputs must be bfloat16 or float16, got {q.dtype}")
    return q.dtype


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, dev):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != dev:
        raise ValueError(f"{name} is on {t.device}, expected {dev}")


def _need_out(t: torch.Tensor, name: str, shape, dtype, dev):
    """A caller-given output: the library writes its whole extent, so it
    must be exactly the shape, dtype and device the call produces, and
    contiguous."""
    _need(t, name, dtype, dev)
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _describe(q, k, v, offsets, max_seq_len, bias, mask):
    """Shape struct + bias struct (with the tensors kept alive)."""
    sh = AttnShape()
    keep = []
    if offsets is None:
        if q.dim() != 4:
            raise ValueError("dense q must be [B, H, M, Dqk]")
        B, H, M, Dqk = q.shape
        N, Dv = k.shape[2], v.shape[3]
        if tuple(k.shape) != (B, H, N, Dqk) or tuple(v.shape) != (B, H, N, Dv):
            raise ValueError("k must be [B, H, N, Dqk] and v [B, H, N, Dv]")
        sh.B, sh.H, sh.M, sh.N, sh.Dqk, sh.Dv, sh.T, sh.max_seq_len = B, H, M, N, Dqk, Dv, 0, 0
        out_shape = (B, H, M, Dv)
    else:
        if q.dim() != 3:
            raise ValueError("jagged q must be [H, T, Dqk]")
        if max_seq_len is None:
            raise ValueError("jagged inputs need max_seq_len")
        H, T, Dqk = q.shape
        Dv = v.shape[2]
        if tuple(k.shape) != (H, T, Dqk) or tuple(v.shape) != (H, T, Dv):
            raise ValueError("k must be [H, T, Dqk] and v [H, T, Dv]")
        sh.B, sh.H, sh.M, sh.N, sh.Dqk, sh.Dv = offsets.numel() - 1, H, 0, 0, Dqk, Dv
        sh.T, sh.max_seq_len = T, int(max_seq_len)
        out_shape = (H, T, Dv)
    bs = None
    if bias is not None or mask is not None:
        if offsets is not None:
            raise ValueError("bias / mask are supported for dense inputs only")
        bs = AttnBias()
        full = (sh.B, sh.H, sh.M, sh.N)
        if bias is not None:
            if bias.dtype != torch.float32 or bias.device != q.device:
                raise TypeError("bias must be float32 on the inputs' device")
            be = bias.expand(full)
            bs.bias = be.data_ptr()
            bs.bias_stride = (ctypes.c_int64 * 4)(*be.stride())
            keep.append(be)
        if mask is not None:
            if mask.dtype == torch.bool:
                mask = mask.view(torch.uint8)
            if mask.dtype != torch.uint8 or mask.device != q.device:
                raise TypeError("mask must be bool/uint8 on the inputs' device")
            me = mask.expand(full)
            bs.mask = me.data_ptr()
            bs.mask_stride = (ctypes.c_int64 * 4)(*me.stride())
            keep.append(me)
    return sh, bs, out_shape, keep


def _scale(sm_scale):
    return float("nan") if sm_scale is None else float(sm_scale)


def attn_fwd_jvp(q, k, v, tq, tk, tv, causal: bool = False, sm_scale: Optional[float] = None,
                 offsets: Optional[torch.Tensor] = None, max_seq_len: Optional[int] = None,
                 bias: Optional[torch.Tensor] = None, mask: Optional[torch.Tensor] = None,
                 out=None):
    """Attention forward + JVP in one pass.  Returns (o, to, lse).

    Dense: q, tq [B, H, M, Dqk]; k, tk [B, H, N, Dqk]; v, tv [B, H, N, Dv].
    Jagged: [H, T, D] with int32 ``offsets`` [B + 1] and ``max_seq_len``.
    ``bias`` (fp32) and ``mask`` (bool/uint8, True = attend) broadcast to
    [B, H, M, N].  CPU inputs are copied to the current CUDA device and the
    outputs copied back (the end-to-end path); CUDA inputs stay on device.
    """
    if q.device.type == "cpu":
        return _host_call(attn_fwd_jvp, (q, k, v, tq, tk, tv), dict(
            causal=causal, sm_scale=sm_scale, offsets=offsets, max_seq_len=max_seq_len,
            bias=bias, mask=mask), n_out=3)
    dev = q.device
    dt = _elem_type(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("tq", tq), ("tk", tk), ("tv", tv)):
        _need(t, name, dt, dev)
    if tq.shape != q.shape or tk.shape != k.shape or tv.shape != v.shape:
        raise ValueError("tangents must have the primals' shapes")
    if offsets is not None:
        _need(offsets, "offsets", torch.int32, dev)
    sh, bs, out_shape, keep = _describe(q, k, v, offsets, max_seq_len, bias, mask)
    if out is None:
        o = torch.empty(out_shape, dtype=dt, device=dev)
        to = torch.empty(out_shape, dtype=dt, device=dev)
        lse = torch.empty(out_shape[:-1], dtype=torch.float32, device=dev)
    else:
        o, to, lse = out
        _need_out(o, "o", out_shape, dt, dev)
        _need_out(to, "to", out_shape, dt, dev)
        _need_out(lse, "lse", out_shape[:-1], torch.float32, dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    fn = lib().attn_fwd_jvp_f16 if dt == torch.float16 else lib().attn_fwd_jvp
    st = fn(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(tq), _ptr(tk),
                            _ptr(tv), _ptr(offsets), ctypes.byref(bs) if bs is not None else None,
                            1 if causal else 0, _scale(sm_scale), _ptr(o), _ptr(to), _ptr(lse),
                            ctypes.c_void_p(stream))
    del keep
    _check(st)
    return o, to, lse


def attn_fwd(q, k, v, causal: bool = False, sm_scale: Optional[float] = None,
             offsets: Optional[torch.Tensor] = None, max_seq_len: Optional[int] = None,
             bias: Optional[torch.Tensor] = None, mask: Optional[torch.Tensor] = None, out=None):
    """Attention forward only.  Returns (o, lse)."""
    if q.device.type == "cpu":
        return _host_call(attn_fwd, (q, k, v), dict(
            causal=causal, sm_scale=sm_scale, offsets=offsets, max_seq_len=max_seq_len,
            bias=bias, mask=mask), n_out=2)
    dev = q.device
    dt = _elem_type(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, dt, dev)
    if offsets is not None:
        _need(offsets, "offsets", torch.int32, dev)
    sh, bs, out_shape, keep = _describe(q, k, v, offsets, max_seq_len, bias, mask)
    if out is None:
        o = torch.empty(out_shape, dtype=dt, device=dev)
        lse = torch.empty(out_shape[:-1], dtype=torch.float32, device=dev)
    else:
        o, lse = out
        _need_out(o, "o", out_shape, dt, dev)
        _need_out(lse, "lse", out_shape[:-1], torch.float32, dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    fn = lib().attn_fwd_f16 if dt == torch.float16 else lib().attn_fwd
    st = fn(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(offsets),
                        ctypes.byref(bs) if bs is not None else None, 1 if causal else 0,
                        _scale(sm_scale), _ptr(o), _ptr(lse), ctypes.c_void_p(stream))
    del keep
    _check(st)
    return o, lse


BWD_DELTA, BWD_DQ, BWD_DKDV, BWD_ALL = 1, 2, 4, 7


def attn_bwd(q, k, v, o, lse, do, causal: bool = False, sm_scale: Optional[float] = None,
             offsets: Optional[torch.Tensor] = None, max_seq_len: Optional[int] = None,
             bias: Optional[torch.Tensor] = None, mask: Optional[torch.Tensor] = None,
             out=None, stages: int = BWD_ALL):
    """Attention backward.  Takes the forward's inputs (with its ``bias`` /
    ``mask``, dense only; the bias gets no gradient), its output ``o`` and
    log-sum-exp ``lse`` and the gradient ``do`` of O; returns
    (dq, dk, dv, delta), delta = rowsum(do o o) in float32.  Dense
    ``[B, H, M|N, D]`` or jagged ``[H, T, D]`` with int32 ``offsets`` and
    ``max_seq_len`` (tokens past a sequence's cap get zero gradients).
    ``stages`` (an OR of BWD_DELTA, BWD_DQ, BWD_DKDV) runs a subset of the
    launches; the others leave their outputs as given."""
    if q.device.type == "cpu":
        return _host_call(attn_bwd, (q, k, v, o, lse, do),
                          dict(causal=causal, sm_scale=sm_scale, offsets=offsets,
                               max_seq_len=max_seq_len, bias=bias, mask=mask), n_out=4)
    dev = q.device
    dt = _elem_type(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _need(t, name, dt, dev)
    _need(lse, "lse", torch.float32, dev)
    if offsets is not None:
        _need(offsets, "offsets", torch.int32, dev)
    sh, bs, out_shape, keep = _describe(q, k, v, offsets, max_seq_len, bias, mask)
    if tuple(o.shape) != out_shape or tuple(do.shape) != out_shape or tuple(lse.shape) != out_shape[:-1]:
        raise ValueError("o and do must be shaped like the forward's output and lse like its log-sum-exp")
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        delta = torch.empty(out_shape[:-1], dtype=torch.float32, device=dev)
    else:
        dq, dk, dv, delta = out
        _need_out(dq, "dq", q.shape, dt, dev)
        _need_out(dk, "dk", k.shape, dt, dev)
        _need_out(dv, "dv", v.shape, dt, dev)
        _need_out(delta, "delta", out_shape[:-1], torch.float32, dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    if stages == BWD_ALL:
        fn = lib().attn_bwd_f16 if dt == torch.float16 else lib().attn_bwd
        st = fn(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(offsets),
                ctypes.byref(bs) if bs is not None else None, 1 if causal else 0, _scale(sm_scale),
                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(delta), ctypes.c_void_p(stream))
    else:
        st = lib().attn_bwd_stages(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do),
                                   _ptr(lse), _ptr(offsets), ctypes.byref(bs) if bs is not None else None,
                                   1 if causal else 0, _scale(sm_scale),
                                   _ptr(dq), _ptr(dk), _ptr(dv), _ptr(delta),
                                   1 if dt == torch.float16 else 0, int(stages), ctypes.c_void_p(stream))
    del keep
    _check(st)
    return dq, dk, dv, delta


def attn_fwd_f8(q, k, vt, causal: bool = False, sm_scale: Optional[float] = None, out=None):
    """FP8 (e5m2) forward: q [B, H, M, D], k [B, H, N, D] and the transposed
    value vt [B, H, D, N], all torch.float8_e5m2.  Returns (o, lse): o e5m2
    [B, H, M, D], lse float32 [B, H, M]."""
    if q.device.type == "cpu":
        return _host_call(attn_fwd_f8, (q, k, vt), dict(causal=causal, sm_scale=sm_scale), n_out=2)
    dev = q.device
    dt = torch.float8_e5m2
    for name, t in (("q", q), ("k", k), ("vt", vt)):
        _need(t, name, dt, dev)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, M, D]")
    B, H, M, D = q.shape
    N = k.shape[2]
    if tuple(k.shape) != (B, H, N, D) or tuple(vt.shape) != (B, H, D, N):
        raise ValueError("k must be [B, H, N, D] and vt [B, H, D, N]")
    sh = AttnShape()
    sh.B, sh.H, sh.M, sh.N, sh.Dqk, sh.Dv, sh.T, sh.max_seq_len = B, H, M, N, D, D, 0, 0
    if out is None:
        o = torch.empty((B, H, M, D), dtype=dt, device=dev)
        lse = torch.empty((B, H, M), dtype=torch.float32, device=dev)
    else:
        o, lse = out
        _need_out(o, "o", (B, H, M, D), dt, dev)
        _need_out(lse, "lse", (B, H, M), torch.float32, dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    st = lib().attn_fwd_f8(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(vt), 1 if causal else 0,
                           _scale(sm_scale), _ptr(o), _ptr(lse), ctypes.c_void_p(stream))
    _check(st)
    return o, lse


_STREAMS = {}


def _chunk_streams(dev, n=4):
    """Streams of the chunked host path (per device, created once)."""
    key = dev.index
    if key not in _STREAMS:
        _STREAMS[key] = [torch.cuda.Stream(dev) for _ in range(n)]
    return _STREAMS[key]


def _slab_chunks(fn, tensors, kw) -> int:
    """How many chunks of whole (batch, head) slabs the host path of a dense
    forward call is cut into: with at least 8 slabs, every tensor contiguous
    and every chunk boundary keeping the 16-byte alignment of the lse rows
    (M a multiple of 4), 4 when the inputs are 128 MB or more and 2 below
    (each chunk costs host time to issue; on a GB300 the copies of a step
    this small finish sooner in two chunks); else 1."""
    if fn not in (attn_fwd_jvp, attn_fwd):
        return 1
    if any(kw.get(k) is not None for k in ("offsets", "bias", "mask")):
        return 1
    q = tensors[0]
    if q.dim() != 4 or any(t.dim() != 4 or t.shape[:2] != q.shape[:2] or not t.is_contiguous()
                           for t in tensors):
        return 1
    if q.shape[0] * q.shape[1] < 8 or q.shape[2] % 4 != 0:
        return 1
    nbytes = sum(t.numel() * t.element_size() for t in tensors)
    return 4 if nbytes >= (128 << 20) else 2


def _host_call(fn, tensors, kw, n_out):
    """End-to-end path for host tensors: copy in, compute, copy out.

    A dense forward without bias or mask is cut into chunks of whole
    (batch, head) slabs, each an independent problem computed by its own
    call of the C entry point (the whole problem is validated once, then
    each chunk passes its slab pointers); a chunk's input copies, kernel and
    output copies run in order on a stream of its own, so the copies of one
    chunk overlap the kernel of another.  The results are those of one call
    over the whole batch."""
    dev = torch.device("cuda", torch.cuda.current_device())
    n = _slab_chunks(fn, tensors, kw)
    if n == 1:
        dt = [t.to(dev, non_blocking=True) for t in tensors]
        for key in ("offsets", "bias", "mask"):
            if kw.get(key) is not None:
                kw[key] = kw[key].to(dev, non_blocking=True)
        outs = fn(*dt, **kw)
        host = tuple(torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs)
        for h, o in zip(host, outs):
            h.copy_(o, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()
        return host[:n_out]

    q, v = tensors[0], tensors[2]
    B, H, M = q.shape[0], q.shape[1], q.shape[2]
    S = B * H
    shapes = [(B, H, M, v.shape[3])] * (n_out - 1) + [(B, H, M)]
    dtypes = [q.dtype] * (n_out - 1) + [torch.float32]
    d_in = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in tensors]
    d_out = [torch.empty(sh, dtype=dt, device=dev) for sh, dt in zip(shapes, dtypes)]
    h_out = [torch.empty(sh, dtype=dt, pin_memory=True) for sh, dt in zip(shapes, dtypes)]

    def slab(t, a, b):  # slabs [a, b) of a [B, H, ...] tensor, as [1, b - a, ...]
        return t.view(S, *t.shape[2:])[a:b].view(1, b - a, *t.shape[2:])

    # the whole problem through the binding's checks once (shapes, dtypes,
    # devices), with no launch: the chunks below skip them
    jvp = fn is attn_fwd_jvp
    f16 = _elem_type(q) == torch.float16
    for name, t in zip(("q", "k", "v", "tq", "tk", "tv"), d_in):
        _need(t, name, q.dtype, dev)
    if jvp and (tensors[3].shape != q.shape or tensors[4].shape != tensors[1].shape
                or tensors[5].shape != v.shape):
        raise ValueError("tangents must have the primals' shapes")
    sh, _, _, _ = _describe(d_in[0], d_in[1], d_in[2], None, None, None, None)
    L = lib()
    cfn = (L.attn_fwd_jvp_f16 if f16 else L.attn_fwd_jvp) if jvp else (L.attn_fwd_f16 if f16 else L.attn_fwd)
    scale = _scale(kw.get("sm_scale"))
    causal = 1 if kw.get("causal") else 0
    per_in = [t.numel() // S * t.element_size() for t in d_in]      # bytes per slab
    per_out = [t.numel() // S * t.element_size() for t in d_out]
    cur = torch.cuda.current_stream(dev)
    streams = _chunk_streams(dev)
    for st in streams:
        st.wait_stream(cur)
    try:
        for c in range(n):
            a, b = S * c // n, S * (c + 1) // n
            st = streams[c % len(streams)]
            with torch.cuda.stream(st):
                for h, d in zip(tensors, d_in):
                    slab(d, a, b).copy_(slab(h, a, b), non_blocking=True)
                csh = AttnShape()
                csh.B, csh.H, csh.M, csh.N, csh.Dqk, csh.Dv = 1, b - a, sh.M, sh.N, sh.Dqk, sh.Dv
                pin = [ctypes.c_void_p(d.data_ptr() + a * pb) for d, pb in zip(d_in, per_in)]
                pout = [ctypes.c_void_p(o.data_ptr() + a * pb) for o, pb in zip(d_out, per_out)]
                # (q, k, v[, tq, tk, tv], offsets, bias, causal, scale, o[, to], lse, stream)
                _check(cfn(ctypes.byref(csh), *pin, None, None, causal, scale, *pout,
                           ctypes.c_void_p(st.cuda_stream)))
                for ho, o in zip(h_out, d_out):
                    slab(ho, a, b).copy_(slab(o, a, b), non_blocking=True)
    finally:
        # also when a chunk's call raises: no copy may still be running
        # when the device buffers are released
        for st in streams:
            st.synchronize()
    return tuple(h_out[:n_out])
