"""Sliding-window attention with a per-head attention sink, on B300 (sm_103a).

Thin Python binding over the C ABI of ``libswasink.so`` (declared in
``include/swasink.h``).  Functions take torch CUDA tensors, check shapes and
dtypes, and pass raw device pointers, sizes and the current CUDA stream to the
library; every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library cannot be loaded, calls raise.

Operation ("MiMo-V2-Flash Technical Report" summary, section 前置知识: hybrid
sliding-window / global attention, a learnable bias added to each head's softmax
denominator; section 核心方法: 128-token window, 5:1 window:global layers):

    out[b,i,h] = sum_{j in [i-W+1, i], j >= 0} exp(x_ij - m) v[b,j,h//G]
                 / (exp(sink[h] - m) + sum_j exp(x_ij - m)),   x_ij = q.k / sqrt(D)
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import inputs, work  # noqa: F401  (host-only helpers)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libswasink.so")

SWA_OK, SWA_EINVAL, SWA_EUNSUPPORTED, SWA_ECUDA = 0, -1, -2, -3
SWA_F32, SWA_BF16 = 0, 1

_lib = None
_lock = threading.Lock()


class SwaError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        msg = f"{fn} failed: {status_str(status)} ({status})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """Load libswasink.so (raises if it is missing or cannot be loaded)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m hybrid_sliding_window_02_b300.build`")
            L = ctypes.CDLL(LIB_PATH)
            p, i32 = ctypes.c_void_p, ctypes.c_int
            L.swa_sink_fwd.argtypes = [p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, p]
            L.swa_sink_fwd_ex.argtypes = [p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32,
                                          p]
            L.swa_sink_fwd_ex.restype = i32
            L.swa_sink_fwd_host.argtypes = [p] * 11 + [i32] * 8 + [p]
            L.swa_sink_fwd_host.restype = i32
            L.swa_sink_fwd_host_static.argtypes = [p] * 6 + [i32] * 8 + [p]
            L.swa_sink_fwd_host_static.restype = i32
            L.swa_sink_decode.argtypes = [p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, p]
            L.swa_ring_append.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, p]
            L.swa_sink_verify.argtypes = [p, p, p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32,
                                          i32, p]
            dbl = ctypes.c_double
            L.swa_rope.argtypes = [p, p, i32, i32, i32, i32, i32, dbl, i32, p]
            L.swa_rope_append.argtypes = [p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, dbl,
                                          i32, p]
            L.swa_rope.restype = i32
            L.swa_rope_append.restype = i32
            L.swa_sink_fwd_scores.argtypes = [p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32,
                                              i32, i32, p]
            L.swa_topk_blocks.argtypes = [p, p, i32, i32, i32, i32, i32, p]
            L.swa_sink_sparse_fwd.argtypes = [p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32,
                                              i32, i32, i32, p]
            for f in (L.swa_sink_fwd_scores, L.swa_topk_blocks, L.swa_sink_sparse_fwd):
                f.restype = i32
            L.swa_sink_verify_path.argtypes = [i32, i32, i32, i32, i32, i32, i32]
            L.swa_sink_verify_path.restype = ctypes.c_char_p
            for f in (L.swa_sink_fwd, L.swa_sink_decode, L.swa_ring_append, L.swa_sink_verify):
                f.restype = i32
            L.swa_sink_fwd_path.argtypes = [i32, i32, i32, i32, i32, i32, i32]
            L.swa_sink_fwd_path.restype = ctypes.c_char_p
            L.swa_sink_decode_path.argtypes = [i32, i32, i32, i32, i32, i32]
            L.swa_sink_decode_path.restype = ctypes.c_char_p
            L.swa_status_str.argtypes = [i32]
            L.swa_status_str.restype = ctypes.c_char_p
            L.swa_last_error.restype = ctypes.c_char_p
            L.swa_device_error.restype = i32
            L.swa_version.restype = i32
            L.swa_test_withhold_loads.argtypes = [i32]
            L.swa_test_withhold_loads.restype = i32
            _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().swa_status_str(int(status)).decode()


def last_error() -> str:
    return lib().swa_last_error().decode()


def device_error() -> int:
    """Read and clear the device-side error word (synchronises the device)."""
    return int(lib().swa_device_error())


def version() -> int:
    return int(lib().swa_version())


def _check(fn: str, status: int):
    if status != SWA_OK:
        raise SwaError(fn, status, last_error())


def _call(fn: str, dev, *args):
    """Call library entry point ``fn`` with ``dev`` as the current CUDA device:
    the library launches on the current device and looks up its attributes
    there, so the tensors' device must be current during the call."""
    import torch
    with torch.cuda.device(dev):
        status = getattr(lib(), fn)(*args)
    _check(fn, status)


def _out_check(name, t, shape, dtypes, device):
    """A caller-supplied output buffer: a contiguous tensor on ``device`` with
    exactly ``shape`` and one of ``dtypes`` (the kernels write it in full)."""
    _cuda_contig(name, t, device)
    if tuple(t.shape) != tuple(shape) or t.dtype not in dtypes:
        names = " or ".join(str(d).replace("torch.", "") for d in dtypes)
        raise ValueError(f"{name} must be {names} {list(shape)}, got {t.dtype} {list(t.shape)}")


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return SWA_BF16
    if t.dtype == torch.float32:
        return SWA_F32
    raise TypeError(f"unsupported input dtype {t.dtype} (bfloat16 or float32)")


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _cuda_contig(name, t, device=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def fwd_path(B, T, Hq, Hkv, D, W, dtype_code=SWA_BF16) -> str:
    """Name of the prefill kernel the library selects for these sizes."""
    return lib().swa_sink_fwd_path(B, T, Hq, Hkv, D, W, dtype_code).decode()


def decode_path(B, Hq, Hkv, D, W, dtype_code=SWA_BF16) -> str:
    """Name of the decode kernel the library selects for these sizes."""
    return lib().swa_sink_decode_path(B, Hq, Hkv, D, W, dtype_code).decode()


def swa_sink_fwd(q, k, v, sink, W: int, out=None, lse=None, *, with_lse: bool = True,
                 out_dtype=None, stream=None):
    """Prefill.  q [B,T,Hq,D], k/v [B,T,Hkv,D] (bf16 or fp32), sink [Hq] fp32.

    Returns (out [B,T,Hq,D], lse [B,Hq,T] fp32 or None).  W >= T is the global
    (full causal) layer.  out is fp32 unless out_dtype (or a given out) is
    torch.bfloat16, which the tensor-core kernels write rounded from fp32.
    """
    import torch
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v), ("sink", sink)):
        _cuda_contig(n, t, dev)
    if k.shape != (B, T, Hkv, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, T, Hkv, D] matching q")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if sink.dtype != torch.float32 or sink.shape != (Hq,):
        raise ValueError("sink must be float32 [Hq]")
    if out is None:
        out = torch.empty(B, T, Hq, D, dtype=out_dtype or torch.float32, device=dev)
    _out_check("out", out, (B, T, Hq, D), (torch.float32, torch.bfloat16), dev)
    if with_lse and lse is None:
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
    if lse is not None:
        _out_check("lse", lse, (B, Hq, T), (torch.float32,), dev)
    _call("swa_sink_fwd_ex", dev, q.data_ptr(), k.data_ptr(), v.data_ptr(), sink.data_ptr(),
          out.data_ptr(), lse.data_ptr() if lse is not None else None,
          B, T, Hq, Hkv, D, int(W), _dtype_code(q), _dtype_code(out),
          _stream_handle(stream, dev))
    return out, lse


def swa_sink_fwd_host(q_h, k_h, v_h, sink, W: int, out_h=None, lse_h=None, *, work=None,
                      with_lse: bool = True, out_dtype=None, stream=None):
    """Prefill from and to host memory, pipelined in chunks (one sequence x a
    range of positions on the sliding-window tensor-core path, one sequence x
    a share of the kv heads otherwise): the copies of one chunk overlap the
    compute and the copies of its neighbours.

    q_h [B,T,Hq,D], k_h/v_h [B,T,Hkv,D]: CPU tensors (pin them for overlap);
    sink [Hq] fp32 on the device.  work: optional tuple of device buffers
    (q_d, k_d, v_d, out_d, lse_d) of the full sizes, reused across calls;
    allocated here when omitted.  Returns (out_h, lse_h or None, work).  The
    host outputs are complete once the stream has been synchronised.
    """
    import torch
    B, T, Hq, D = q_h.shape
    Hkv = k_h.shape[2]
    for n, t in (("q_h", q_h), ("k_h", k_h), ("v_h", v_h)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU tensor")
    if k_h.shape != (B, T, Hkv, D) or v_h.shape != k_h.shape:
        raise ValueError("k_h and v_h must be [B, T, Hkv, D] matching q_h")
    if k_h.dtype != q_h.dtype or v_h.dtype != q_h.dtype:
        raise TypeError("q, k, v must share one dtype")
    if sink.dtype != torch.float32 or sink.shape != (Hq,):
        raise ValueError("sink must be float32 [Hq]")
    dev = sink.device
    _cuda_contig("sink", sink, dev)
    odt = out_dtype or (out_h.dtype if out_h is not None else torch.float32)
    pin = q_h.is_pinned()
    if out_h is None:
        out_h = torch.empty(B, T, Hq, D, dtype=odt, pin_memory=pin)
    if with_lse and lse_h is None:
        lse_h = torch.empty(B, Hq, T, dtype=torch.float32, pin_memory=pin)
    _host_out_check(out_h, lse_h, B, T, Hq, D)
    if work is None:
        work = (torch.empty(q_h.shape, dtype=q_h.dtype, device=dev),
                torch.empty(k_h.shape, dtype=k_h.dtype, device=dev),
                torch.empty(v_h.shape, dtype=v_h.dtype, device=dev),
                torch.empty(out_h.shape, dtype=out_h.dtype, device=dev),
                torch.empty(B, Hq, T, dtype=torch.float32, device=dev) if lse_h is not None
                else None)
    q_d, k_d, v_d, out_d, lse_d = work
    for n, t, ref in (("q_d", q_d, q_h), ("k_d", k_d, k_h), ("v_d", v_d, v_h),
                      ("out_d", out_d, out_h)):
        _cuda_contig(n, t, dev)
        if t.shape != ref.shape or t.dtype != ref.dtype:
            raise ValueError(f"{n} must match {tuple(ref.shape)} {ref.dtype}")
    if (lse_h is None) != (lse_d is None):
        raise ValueError("lse_h and lse_d go together")
    if lse_d is not None:
        _out_check("lse_d", lse_d, (B, Hq, T), (torch.float32,), dev)
    _call("swa_sink_fwd_host", dev, q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(),
          sink.data_ptr(), out_h.data_ptr(), lse_h.data_ptr() if lse_h is not None else None,
          q_d.data_ptr(), k_d.data_ptr(), v_d.data_ptr(), out_d.data_ptr(),
          lse_d.data_ptr() if lse_d is not None else None,
          B, T, Hq, Hkv, D, int(W), _dtype_code(q_h), _dtype_code(out_h),
          _stream_handle(stream, dev))
    return out_h, lse_h, work


def _host_out_check(out_h, lse_h, B, T, Hq, D):
    """Host outputs of the host-memory prefill: contiguous CPU tensors, out_h
    [B, T, Hq, D] fp32 or bf16, lse_h [B, Hq, T] fp32 (or None)."""
    import torch
    if (out_h.is_cuda or tuple(out_h.shape) != (B, T, Hq, D) or not out_h.is_contiguous()
            or out_h.dtype not in (torch.float32, torch.bfloat16)):
        raise ValueError("out_h must be a contiguous CPU tensor [B, T, Hq, D], float32 or "
                         "bfloat16")
    if lse_h is not None and (lse_h.is_cuda or tuple(lse_h.shape) != (B, Hq, T) or
                              lse_h.dtype != torch.float32 or not lse_h.is_contiguous()):
        raise ValueError("lse_h must be a contiguous CPU float32 tensor [B, Hq, T]")


def swa_sink_fwd_host_static(q_h, k_h, v_h, sink, W: int, out_h=None, lse_h=None, *,
                             with_lse: bool = True, out_dtype=None, stream=None):
    """swa_sink_fwd_host for callers that cannot allocate device memory: the
    data in transit goes through the library's own static staging array
    (SWA_HOST_STATIC_BYTES per GPU), so no device buffer is passed or made.
    Raises SwaError (unsupported) when the sizes need more staging than that.
    Calls whose GPU work overlaps share the array and race; order them on one
    stream.  Returns (out_h, lse_h or None), complete once the stream has been
    synchronised."""
    import torch
    B, T, Hq, D = q_h.shape
    Hkv = k_h.shape[2]
    for n, t in (("q_h", q_h), ("k_h", k_h), ("v_h", v_h)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU tensor")
    if k_h.shape != (B, T, Hkv, D) or v_h.shape != k_h.shape:
        raise ValueError("k_h and v_h must be [B, T, Hkv, D] matching q_h")
    if k_h.dtype != q_h.dtype or v_h.dtype != q_h.dtype:
        raise TypeError("q, k, v must share one dtype")
    if sink.dtype != torch.float32 or sink.shape != (Hq,):
        raise ValueError("sink must be float32 [Hq]")
    dev = sink.device
    _cuda_contig("sink", sink, dev)
    odt = out_dtype or (out_h.dtype if out_h is not None else torch.float32)
    pin = q_h.is_pinned()
    if out_h is None:
        out_h = torch.empty(B, T, Hq, D, dtype=odt, pin_memory=pin)
    if with_lse and lse_h is None:
        lse_h = torch.empty(B, Hq, T, dtype=torch.float32, pin_memory=pin)
    _host_out_check(out_h, lse_h, B, T, Hq, D)
    _call("swa_sink_fwd_host_static", dev, q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(),
          sink.data_ptr(), out_h.data_ptr(), lse_h.data_ptr() if lse_h is not None else None,
          B, T, Hq, Hkv, D, int(W), _dtype_code(q_h), _dtype_code(out_h),
          _stream_handle(stream, dev))
    return out_h, lse_h


def swa_sink_decode(q, k_ring, v_ring, pos, sink, out=None, lse=None, *, with_lse=True,
                    stream=None):
    """Decode.  q [B,Hq,D], rings [B,Hkv,W,D], pos [B] int64, sink [Hq] fp32.

    Returns (out [B,Hq,D] fp32, lse [B,Hq] fp32 or None).
    """
    import torch
    B, Hq, D = q.shape
    _, Hkv, W, _ = k_ring.shape
    dev = q.device
    for n, t in (("q", q), ("k_ring", k_ring), ("v_ring", v_ring), ("pos", pos),
                 ("sink", sink)):
        _cuda_contig(n, t, dev)
    if k_ring.shape != (B, Hkv, W, D) or v_ring.shape != k_ring.shape:
        raise ValueError("rings must be [B, Hkv, W, D] matching q")
    if pos.dtype != torch.int64 or pos.shape != (B,):
        raise ValueError("pos must be int64 [B]")
    if k_ring.dtype != q.dtype or v_ring.dtype != q.dtype:
        raise TypeError("q and rings must share one dtype")
    if sink.dtype != torch.float32 or sink.shape != (Hq,):
        raise ValueError("sink must be float32 [Hq]")
    if out is None:
        out = torch.empty(B, Hq, D, dtype=torch.float32, device=dev)
    _out_check("out", out, (B, Hq, D), (torch.float32,), dev)
    if with_lse and lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    if lse is not None:
        _out_check("lse", lse, (B, Hq), (torch.float32,), dev)
    _call("swa_sink_decode", dev, q.data_ptr(), k_ring.data_ptr(), v_ring.data_ptr(),
          pos.data_ptr(), sink.data_ptr(), out.data_ptr(),
          lse.data_ptr() if lse is not None else None,
          B, Hq, Hkv, D, W, _dtype_code(q), _stream_handle(stream, dev))
    return out, lse


def verify_path(B, L, Hq, Hkv, D, W, dtype_code=SWA_BF16) -> str:
    """Name of the verify kernel the library selects for these sizes."""
    return lib().swa_sink_verify_path(B, L, Hq, Hkv, D, W, dtype_code).decode()


def swa_sink_verify(q, k_new, v_new, k_ring, v_ring, pos, sink, out=None, lse=None, *,
                    with_lse=True, stream=None):
    """Multi-token verify.  q [B,L,Hq,D], k_new/v_new [B,L,Hkv,D] (the drafted
    tokens), rings [B,Hkv,W,D] holding the positions before pos, pos [B] int64
    (position of drafted token 0), sink [Hq] fp32.

    Returns (out [B,L,Hq,D] fp32, lse [B,Hq,L] fp32 or None).
    """
    import torch
    B, L, Hq, D = q.shape
    _, Hkv, W, _ = k_ring.shape
    dev = q.device
    for n, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("k_ring", k_ring),
                 ("v_ring", v_ring), ("pos", pos), ("sink", sink)):
        _cuda_contig(n, t, dev)
    if k_new.shape != (B, L, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must be [B, L, Hkv, D] matching q")
    if k_ring.shape != (B, Hkv, W, D) or v_ring.shape != k_ring.shape:
        raise ValueError("rings must be [B, Hkv, W, D] matching q")
    if pos.dtype != torch.int64 or pos.shape != (B,):
        raise ValueError("pos must be int64 [B]")
    for n, t in (("k_new", k_new), ("v_new", v_new), ("k_ring", k_ring), ("v_ring", v_ring)):
        if t.dtype != q.dtype:
            raise TypeError(f"{n} must have the dtype of q")
    if sink.dtype != torch.float32 or sink.shape != (Hq,):
        raise ValueError("sink must be float32 [Hq]")
    if out is None:
        out = torch.empty(B, L, Hq, D, dtype=torch.float32, device=dev)
    _out_check("out", out, (B, L, Hq, D), (torch.float32,), dev)
    if with_lse and lse is None:
        lse = torch.empty(B, Hq, L, dtype=torch.float32, device=dev)
    if lse is not None:
        _out_check("lse", lse, (B, Hq, L), (torch.float32,), dev)
    _call("swa_sink_verify", dev, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
          k_ring.data_ptr(), v_ring.data_ptr(), pos.data_ptr(), sink.data_ptr(), out.data_ptr(),
          lse.data_ptr() if lse is not None else None,
          B, L, Hq, Hkv, D, W, _dtype_code(q), _stream_handle(stream, dev))
    return out, lse


def swa_rope(x, pos0, rot_dim: int, theta: float, *, stream=None):
    """Rotary embedding in place on x [B,T,H,D] (bf16 or fp32); token (b, t)
    is at position pos0[b] + t (pos0 int64 [B] on the device).  Returns x."""
    import torch
    B, T, H, D = x.shape
    dev = x.device
    _cuda_contig("x", x, dev)
    _cuda_contig("pos0", pos0, dev)
    if pos0.dtype != torch.int64 or pos0.shape != (B,):
        raise ValueError("pos0 must be int64 [B]")
    _call("swa_rope", dev, x.data_ptr(), pos0.data_ptr(), B, T, H, D, int(rot_dim),
          float(theta), _dtype_code(x), _stream_handle(stream, dev))
    return x


def swa_rope_append(q, k, v, k_ring, v_ring, pos, rot_dim: int, theta: float, q_out=None, *,
                    stream=None):
    """Rotate the new token's q [B,Hq,D] and k [B,Hkv,D] at pos [B] and write k,
    v [B,Hkv,D] into ring slot pos mod W of k_ring / v_ring [B,Hkv,W,D].
    Returns the rotated q (q_out, a new tensor unless given; may be q)."""
    import torch
    B, Hq, D = q.shape
    _, Hkv, W, _ = k_ring.shape
    dev = q.device
    if q_out is None:
        q_out = torch.empty_like(q)
    for n, t in (("q", q), ("k", k), ("v", v), ("k_ring", k_ring), ("v_ring", v_ring),
                 ("pos", pos), ("q_out", q_out)):
        _cuda_contig(n, t, dev)
    if (k.shape != (B, Hkv, D) or v.shape != k.shape or k_ring.shape != (B, Hkv, W, D)
            or v_ring.shape != k_ring.shape or q_out.shape != q.shape):
        raise ValueError("shape mismatch between q, q_out, the new tokens and the rings")
    if pos.dtype != torch.int64 or pos.shape != (B,):
        raise ValueError("pos must be int64 [B]")
    for n, t in (("k", k), ("v", v), ("k_ring", k_ring), ("v_ring", v_ring), ("q_out", q_out)):
        if t.dtype != q.dtype:
            raise TypeError(f"{n} must have the dtype of q")
    _call("swa_rope_append", dev, q.data_ptr(), k.data_ptr(), v.data_ptr(), q_out.data_ptr(),
          k_ring.data_ptr(), v_ring.data_ptr(), pos.data_ptr(), B, Hq, Hkv, D, W, int(rot_dim),
          float(theta), _dtype_code(q), _stream_handle(stream, dev))
    return q_out


def _prefill_checks(q, k, v, sink):
    import torch
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v), ("sink", sink)):
        _cuda_contig(n, t, dev)
    if k.shape != (B, T, Hkv, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, T, Hkv, D] matching q")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if sink.dtype != torch.float32 or sink.shape != (Hq,):
        raise ValueError("sink must be float32 [Hq]")
    return B, T, Hq, Hkv, D, dev


def swa_sink_fwd_scores(q, k, v, sink, W: int, *, out_dtype=None, stream=None):
    """Prefill on the tensor-core global kernel that also returns the block
    scores of High Sparse: (out, lse, blockmax [B, Hkv, ceil(T/4), ceil(T/128)]
    fp32, -inf where a block holds no valid pair)."""
    import torch
    B, T, Hq, Hkv, D, dev = _prefill_checks(q, k, v, sink)
    out = torch.empty(B, T, Hq, D, dtype=out_dtype or torch.float32, device=dev)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
    bm = torch.full((B, Hkv, (T + 3) // 4, (T + 127) // 128), float("-inf"),
                    dtype=torch.float32, device=dev)
    _call("swa_sink_fwd_scores", dev, q.data_ptr(), k.data_ptr(), v.data_ptr(),
          sink.data_ptr(), out.data_ptr(), lse.data_ptr(), bm.data_ptr(), B, T, Hq, Hkv, D,
          int(W), _dtype_code(q), _dtype_code(out), _stream_handle(stream, dev))
    return out, lse, bm


def swa_topk_blocks(scores, T: int, QB: int, topk: int, *, stream=None):
    """Block selection: int32 [B, Hkv, ceil(T/QB), topk], increasing, -1 padded."""
    import torch
    B, Hkv = scores.shape[0], scores.shape[1]
    dev = scores.device
    _cuda_contig("scores", scores, dev)
    if scores.dtype != torch.float32 or scores.shape != (B, Hkv, (T + 3) // 4, (T + 127) // 128):
        raise ValueError("scores must be float32 [B, Hkv, ceil(T/4), ceil(T/128)]")
    idx = torch.empty(B, Hkv, (T + QB - 1) // QB, topk, dtype=torch.int32, device=dev)
    _call("swa_topk_blocks", dev, scores.data_ptr(), idx.data_ptr(), B, int(T), Hkv,
          int(QB), int(topk), _stream_handle(stream, dev))
    return idx


def swa_sink_sparse_fwd(q, k, v, sink, idx, QB: int, *, out_dtype=None, stream=None):
    """A sparse layer: causal attention over the key blocks idx selects per
    query block of QB positions.  Returns (out, lse)."""
    import torch
    B, T, Hq, Hkv, D, dev = _prefill_checks(q, k, v, sink)
    _cuda_contig("idx", idx, dev)
    if idx.dtype != torch.int32 or idx.dim() != 4 or idx.shape[:3] != (B, Hkv, (T + QB - 1) // QB):
        raise ValueError("idx must be int32 [B, Hkv, ceil(T/QB), topk]")
    out = torch.empty(B, T, Hq, D, dtype=out_dtype or torch.float32, device=dev)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
    _call("swa_sink_sparse_fwd", dev, q.data_ptr(), k.data_ptr(), v.data_ptr(),
          sink.data_ptr(), idx.data_ptr(), out.data_ptr(), lse.data_ptr(), B, T, Hq, Hkv, D,
          int(QB), int(idx.shape[3]), _dtype_code(q), _dtype_code(out),
          _stream_handle(stream, dev))
    return out, lse


def swa_ring_append(k_new, v_new, k_ring, v_ring, pos, *, stream=None):
    """Write k_new/v_new [B,Hkv,D] into ring slot pos mod W of k_ring/v_ring [B,Hkv,W,D]."""
    import torch
    B, Hkv, W, D = k_ring.shape
    dev = k_ring.device
    for n, t in (("k_new", k_new), ("v_new", v_new), ("k_ring", k_ring), ("v_ring", v_ring),
                 ("pos", pos)):
        _cuda_contig(n, t, dev)
    if k_new.shape != (B, Hkv, D) or v_new.shape != k_new.shape or v_ring.shape != k_ring.shape:
        raise ValueError("shape mismatch between new tokens and rings")
    if pos.dtype != torch.int64 or pos.shape != (B,):
        raise ValueError("pos must be int64 [B]")
    for n, t in (("k_new", k_new), ("v_new", v_new), ("v_ring", v_ring)):
        if t.dtype != k_ring.dtype:
            raise TypeError(f"{n} must have the dtype of k_ring")
    _call("swa_ring_append", dev, k_new.data_ptr(), v_new.data_ptr(), k_ring.data_ptr(),
          v_ring.data_ptr(), pos.data_ptr(), B, Hkv, D, W, _dtype_code(k_ring),
          _stream_handle(stream, dev))
