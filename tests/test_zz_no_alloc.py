"""swa_sink_fwd_host_static: the host-memory prefill for callers that cannot
allocate device memory (their device memory belongs to another allocator, or
their loop must not call cudaMalloc / cudaFree, which can synchronise the
device).  It stages the data in transit in the library's own static array
instead of device buffers from the caller.

The GPU test calls the entry point through the C ABI twice in a row, on
different inputs, and checks each result against swa_sink_fwd_host (the call
with caller-owned staging) on the same inputs.  This file is named to be
collected last, so that a run stopping at the first failure has run every
other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import build as swabuild
from hybrid_sliding_window_02_b300 import inputs as gen

STATIC_BYTES = 64 * 1024 * 1024     # SWA_HOST_STATIC_BYTES in include/swasink.h


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _static_call(x, W, out_h, lse_h, stream):
    """One call of the entry point through the C ABI (ctypes), no binding."""
    B, T, Hq, D = x.q.shape
    Hkv = x.k.shape[2]
    code = swa.SWA_BF16 if x.q.dtype == torch.bfloat16 else swa.SWA_F32
    ocode = swa.SWA_BF16 if out_h.dtype == torch.bfloat16 else swa.SWA_F32
    return swa.lib().swa_sink_fwd_host_static(
        _ptr(x.q), _ptr(x.k), _ptr(x.v), _ptr(x.sink), _ptr(out_h), _ptr(lse_h),
        B, T, Hq, Hkv, D, W, code, ocode, ctypes.c_void_p(stream.cuda_stream))


def _close(got, want, max_abs=2e-2, mean_abs=2e-3):
    d = (got.double() - want.double()).abs()
    assert torch.isfinite(got).all()
    assert d.max().item() <= max_abs and d.mean().item() <= mean_abs, (d.max(), d.mean())


@pytest.mark.gpu
def test_static_staging_call_equals_host_call_twice(cuda_ok):
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    # call 1: sliding-window tensor-core path, two chunks of positions with a
    # ragged tail (53,504 bytes of staging per position); call 2: other inputs
    # and sizes on the global-layer path (chunks by kv heads)
    cases = [(1, 1100, 64, 8, 128, 128, 11), (2, 700, 16, 2, 128, 700, 12)]
    for B, T, Hq, Hkv, D, W, seed in cases:
        x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=seed)
        xs = gen.PrefillInputs(x.q.pin_memory(), x.k.pin_memory(), x.v.pin_memory(),
                               x.sink.to(dev))
        out_h = torch.full((B, T, Hq, D), float("nan"), dtype=torch.float32).pin_memory()
        lse_h = torch.full((B, Hq, T), float("nan"), dtype=torch.float32).pin_memory()
        st = _static_call(xs, W, out_h, lse_h, stream)
        assert st == swa.SWA_OK, (st, swa.last_error())
        stream.synchronize()
        want_o, want_l, _ = swa.swa_sink_fwd_host(xs.q, xs.k, xs.v, xs.sink, W, stream=stream)
        stream.synchronize()
        _close(out_h, want_o)
        d_lse = (lse_h.double() - want_l.double()).abs().max().item()
        assert torch.isfinite(lse_h).all() and d_lse <= 1e-3, d_lse
        # the same kernels on the same data: the results agree bit for bit
        assert torch.equal(out_h, want_o) and torch.equal(lse_h, want_l)
    assert swa.device_error() == 0


def test_static_staging_rejects_sizes_beyond_its_capacity():
    """Sizes whose staging exceeds the static array are refused on the host,
    before any CUDA call (so this runs without a GPU)."""
    swabuild.build()
    L = swa.lib()
    buf = (ctypes.c_char * 64)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    # bf16 in, fp32 out + lse, Hq 64, Hkv 8, D 128: 53,504 bytes per position
    per_pos = 64 * 128 * 2 + 2 * 8 * 128 * 2 + 64 * 128 * 4 + 64 * 4
    fits = STATIC_BYTES // per_pos - 8           # room for the 256-byte roundings
    too_many = STATIC_BYTES // per_pos + 1
    st = L.swa_sink_fwd_host_static(p, p, p, p, p, p, 1, too_many, 64, 8, 128, 128,
                                    swa.SWA_BF16, swa.SWA_F32, None)
    assert st == swa.SWA_EUNSUPPORTED
    assert "static staging" in swa.last_error()
    # without lse the same size needs less staging, still too much at 2 sequences
    st = L.swa_sink_fwd_host_static(p, p, p, p, p, None, 2, fits, 64, 8, 128, 128,
                                    swa.SWA_BF16, swa.SWA_F32, None)
    assert st == swa.SWA_EUNSUPPORTED
    # sizes whose byte counts overflow 64 bits are refused the same way
    st = L.swa_sink_fwd_host_static(p, p, p, p, p, p, 2**31 - 1, 2**31 - 1, 2**30, 2**30,
                                    128, 128, swa.SWA_BF16, swa.SWA_F32, None)
    assert st == swa.SWA_EUNSUPPORTED
    # invalid arguments are caught first
    assert L.swa_sink_fwd_host_static(None, p, p, p, p, p, 1, 16, 64, 8, 128, 128,
                                      swa.SWA_BF16, swa.SWA_F32, None) == swa.SWA_EINVAL
    assert L.swa_sink_fwd_host_static(p, p, p, p, p, p, 1, 16, 64, 7, 128, 128,
                                      swa.SWA_BF16, swa.SWA_F32, None) == swa.SWA_EINVAL
    assert np.isfinite(per_pos) and fits > 1000
