"""CPU fp64 oracle for sliding-window attention with a per-head sink bias.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library path never
does.  It shares no code with the CUDA kernels: the arithmetic lives in
``swa_oracle.c`` (plain C, fp64, OpenMP over rows), which this module compiles
with gcc on first use and calls through ctypes.

Every function follows the definition quoted in ``swa_oracle.c``:
sliding-window causal attention (window W, W >= T = global layer) with GQA and
a learnable per-head bias added to the softmax denominator ("MiMo-V2-Flash
Technical Report" summary, section 前置知识: 混合注意力机制, 注意力sink偏置),
one-token decode against a W-slot ring cache ("pwwt.cn" MiMo-V2-Flash essay,
section 1.1: fixed-size sliding-window KV cache), and the multi-token verify of
drafted tokens against that ring.

Pins (what ties these functions to something other than themselves) live in
``tests/test_oracle_pins.py``: brute force with explicit score matrices, the
sink -> -inf / +inf limits, W >= T against a library causal-attention routine,
weights + sink summing to one, the closed form at W = 1, decode = prefill row,
verify = prefill rows, and poisoned out-of-window keys.  RoPE's frequency
schedule and pair layout are pinned by hand-derived cos/sin values in
``tests/golden/rope_hand_derived.json`` (``tests/test_golden.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_swa.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile swa_oracle.c into liboracle_swa.so (gcc, -O2, OpenMP, IEEE math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.oracle_swa_sink_fwd.argtypes = [p, p, p, p, p, p, i64, i64, i32, i32, i32, i64,
                                                i32, i32]
            lib.oracle_swa_sink_fwd_rows.argtypes = [p, p, p, p, p, i64, p, p, i64, i64, i32,
                                                     i32, i32, i64, i32, i32]
            lib.oracle_swa_sink_decode.argtypes = [p, p, p, p, p, p, p, i64, i32, i32, i32, i64,
                                                   i32, i32]
            lib.oracle_swa_sink_verify.argtypes = [p, p, p, p, p, p, p, p, p, i64, i64, i32, i32,
                                                   i32, i64, i32, i32]
            lib.oracle_rope.argtypes = [p, p, p, i64, i64, i32, i32, i32, ctypes.c_double, i32]
            lib.oracle_block_max.argtypes = [p, p, p, i64, i64, i32, i32, i32, i64, i32, i32]
            lib.oracle_topk_blocks.argtypes = [p, p, i64, i64, i32, i32, i32]
            lib.oracle_sparse_fwd.argtypes = [p, p, p, p, p, p, p, i64, i64, i32, i32, i32, i32,
                                              i32, i32, i32]
            for f in (lib.oracle_block_max, lib.oracle_topk_blocks, lib.oracle_sparse_fwd):
                f.restype = i32
            for f in (lib.oracle_swa_sink_fwd, lib.oracle_swa_sink_fwd_rows,
                      lib.oracle_swa_sink_decode, lib.oracle_swa_sink_verify, lib.oracle_rope):
                f.restype = i32
            lib.oracle_num_threads.restype = i32
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _as_storage(x):
    """Return (contiguous numpy array, dtype code) holding x's stored values.

    torch bf16 tensors are passed as their raw 16-bit patterns; fp32 / fp64 as is.
    """
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            if x.dtype == torch.float64:
                return x.numpy(), F64
            raise TypeError(f"unsupported dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.float64:
        return x, F64
    raise TypeError(f"unsupported dtype {x.dtype}")


def _same_type(*arrs):
    conv = [_as_storage(a) for a in arrs]
    codes = {c for _, c in conv}
    if len(codes) != 1:
        raise TypeError("q, k, v must share one storage type")
    return [a for a, _ in conv], codes.pop()


def _sink64(sink):
    try:
        import torch
        if isinstance(sink, torch.Tensor):
            sink = sink.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(sink, dtype=np.float64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def swa_sink_fwd(q, k, v, sink, W: int, nthreads: int = 0):
    """Prefill oracle.  q [B,T,Hq,D], k/v [B,T,Hkv,D], sink [Hq].

    Returns (out [B,T,Hq,D] float64, lse [B,Hq,T] float64).  W >= T gives the
    global (full causal) layer.
    """
    (qa, ka, va), code = _same_type(q, k, v)
    B, T, Hq, D = qa.shape
    Hkv = ka.shape[2]
    s = _sink64(sink)
    out = np.empty((B, T, Hq, D), dtype=np.float64)
    lse = np.empty((B, Hq, T), dtype=np.float64)
    rc = _load().oracle_swa_sink_fwd(_ptr(qa), _ptr(ka), _ptr(va), _ptr(s), _ptr(out), _ptr(lse),
                                     B, T, Hq, Hkv, D, int(W), code, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_swa_sink_fwd failed ({rc})")
    return out, lse


def swa_sink_fwd_rows(q, k, v, sink, W: int, rows, nthreads: int = 0):
    """Prefill oracle on selected rows.  rows: int array [n, 3] of (b, h, i).

    Returns (out_rows [n, D] float64, lse_rows [n] float64).
    """
    (qa, ka, va), code = _same_type(q, k, v)
    B, T, Hq, D = qa.shape
    Hkv = ka.shape[2]
    s = _sink64(sink)
    sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = sel.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().oracle_swa_sink_fwd_rows(_ptr(qa), _ptr(ka), _ptr(va), _ptr(s), _ptr(sel), n,
                                          _ptr(out), _ptr(lse), B, T, Hq, Hkv, D, int(W), code,
                                          int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_swa_sink_fwd_rows failed ({rc})")
    return out, lse


def _pos64(pos):
    try:
        import torch
        if isinstance(pos, torch.Tensor):
            pos = pos.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(pos, dtype=np.int64)


def swa_sink_verify(q, k_new, v_new, k_ring, v_ring, pos, sink, nthreads: int = 0):
    """Multi-token verify oracle.  q [B,L,Hq,D], k_new/v_new [B,L,Hkv,D],
    rings [B,Hkv,W,D] holding the positions before pos, pos [B] int64 = the
    position of new token 0, sink [Hq].

    Returns (out [B,L,Hq,D] float64, lse [B,Hq,L] float64).
    """
    (qa, kna, vna, kra, vra), code = _same_type(q, k_new, v_new, k_ring, v_ring)
    B, L, Hq, D = qa.shape
    Hkv, W = kra.shape[1], kra.shape[2]
    pa = _pos64(pos)
    s = _sink64(sink)
    out = np.empty((B, L, Hq, D), dtype=np.float64)
    lse = np.empty((B, Hq, L), dtype=np.float64)
    rc = _load().oracle_swa_sink_verify(_ptr(qa), _ptr(kna), _ptr(vna), _ptr(kra), _ptr(vra),
                                        _ptr(pa), _ptr(s), _ptr(out), _ptr(lse), B, L, Hq, Hkv,
                                        D, W, code, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_swa_sink_verify failed ({rc})")
    return out, lse


def rope(x, pos0, rot_dim: int, theta: float):
    """Rotary embedding of x [B,T,H,D] (token (b, t) at position pos0[b] + t),
    rotate-half form over the first rot_dim dims.  Returns float64 [B,T,H,D]."""
    (xa,), code = _same_type(x)
    B, T, H, D = xa.shape
    pa = _pos64(pos0)
    y = np.empty((B, T, H, D), dtype=np.float64)
    rc = _load().oracle_rope(_ptr(xa), _ptr(pa), _ptr(y), B, T, H, D, int(rot_dim),
                             float(theta), code)
    if rc != 0:
        raise ValueError(f"oracle_rope failed ({rc})")
    return y


def block_max(q, k, W: int, nthreads: int = 0):
    """Block scores of a layer: [B, Hkv, ceil(T/4), ceil(T/128)] float64, the max
    scaled logit over the valid pairs of each (kv head, 4-position query group,
    128-key block); -inf where there is none."""
    (qa, ka), code = _same_type(q, k)
    B, T, Hq, D = qa.shape
    Hkv = ka.shape[2]
    out = np.empty((B, Hkv, (T + 3) // 4, (T + 127) // 128), dtype=np.float64)
    rc = _load().oracle_block_max(_ptr(qa), _ptr(ka), _ptr(out), B, T, Hq, Hkv, D, int(W), code,
                                  int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_block_max failed ({rc})")
    return out


def topk_blocks(scores, T: int, QB: int, topk: int):
    """Block selection from scores [B, Hkv, ceil(T/4), ceil(T/128)] (cast to
    float32): int32 [B, Hkv, ceil(T/QB), topk], increasing, padded with -1."""
    sc = np.ascontiguousarray(np.asarray(scores, dtype=np.float32))
    B, Hkv = sc.shape[0], sc.shape[1]
    out = np.empty((B, Hkv, (T + QB - 1) // QB, topk), dtype=np.int32)
    rc = _load().oracle_topk_blocks(_ptr(sc), _ptr(out), B, int(T), Hkv, int(QB), int(topk))
    if rc != 0:
        raise ValueError(f"oracle_topk_blocks failed ({rc})")
    return out


def sparse_fwd(q, k, v, sink, idx, QB: int, nthreads: int = 0):
    """Attention over the selected key blocks: idx [B, Hkv, ceil(T/QB), topk]
    int32.  Returns (out [B,T,Hq,D], lse [B,Hq,T]) float64."""
    (qa, ka, va), code = _same_type(q, k, v)
    B, T, Hq, D = qa.shape
    Hkv = ka.shape[2]
    try:
        import torch
        if isinstance(idx, torch.Tensor):
            idx = idx.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    ia = np.ascontiguousarray(idx, dtype=np.int32)
    topk = ia.shape[-1]
    s = _sink64(sink)
    out = np.empty((B, T, Hq, D), dtype=np.float64)
    lse = np.empty((B, Hq, T), dtype=np.float64)
    rc = _load().oracle_sparse_fwd(_ptr(qa), _ptr(ka), _ptr(va), _ptr(s), _ptr(ia), _ptr(out),
                                   _ptr(lse), B, T, Hq, Hkv, D, int(QB), int(topk), code,
                                   int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_sparse_fwd failed ({rc})")
    return out, lse


def swa_sink_decode(q, k_ring, v_ring, pos, sink, nthreads: int = 0):
    """Decode oracle.  q [B,Hq,D], rings [B,Hkv,W,D], pos [B] int64, sink [Hq].

    Returns (out [B,Hq,D] float64, lse [B,Hq] float64).
    """
    (qa, ka, va), code = _same_type(q, k_ring, v_ring)
    B, Hq, D = qa.shape
    Hkv, W = ka.shape[1], ka.shape[2]
    try:
        import torch
        if isinstance(pos, torch.Tensor):
            pos = pos.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    pa = np.ascontiguousarray(pos, dtype=np.int64)
    s = _sink64(sink)
    out = np.empty((B, Hq, D), dtype=np.float64)
    lse = np.empty((B, Hq), dtype=np.float64)
    rc = _load().oracle_swa_sink_decode(_ptr(qa), _ptr(ka), _ptr(va), _ptr(pa), _ptr(s),
                                        _ptr(out), _ptr(lse), B, Hq, Hkv, D, W, code,
                                        int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_swa_sink_decode failed ({rc})")
    return out, lse
