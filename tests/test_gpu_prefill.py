"""GPU prefill parity against the fp64 oracle (element by element)."""
import math

import numpy as np
import pytest
import torch

import oracle
import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen
from gpu_helpers import (assert_bf16_close, assert_f32_close, assert_lse_close, gather_rows,
                         oracle_by_slices, oracle_rows_from_slices, sample_rows)

pytestmark = pytest.mark.gpu


def _run(x, W, dev="cuda"):
    q, k, v, s = (t.to(dev) for t in (x.q, x.k, x.v, x.sink))
    out, lse = swa.swa_sink_fwd(q, k, v, s, W)
    torch.cuda.synchronize()
    return out, lse


def _full_check(x, W, fp32=False):
    out, lse = _run(x, W)
    o_ref, l_ref = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    if fp32:
        assert_f32_close(out.cpu().double().numpy(), o_ref)
        assert_f32_close(lse.cpu().double().numpy(), l_ref, what="lse")
    else:
        assert_bf16_close(out.cpu().numpy(), o_ref)
        assert_lse_close(lse.cpu().numpy(), l_ref)
    return out, lse


# ---- tensor-core sliding-window kernel: small shapes, full comparison -------
@pytest.mark.parametrize("B,T,Hq,Hkv,W", [
    (1, 16, 8, 1, 128),      # one tile
    (1, 1, 8, 1, 128),       # a single position
    (1, 17, 8, 1, 128),      # ragged tail
    (1, 300, 8, 1, 128),
    (2, 200, 16, 2, 128),
    (1, 300, 8, 1, 1),       # window of one key
    (1, 300, 8, 1, 16),
    (1, 300, 8, 1, 100),
    (1, 300, 8, 1, 129),     # largest window of this kernel
    (3, 1000, 16, 2, 128),   # many tiles per CTA, runs crossing CTA boundaries
    (1, 4099, 64, 8, 128),
])
def test_tc_swa_matches_oracle(cuda_ok, B, T, Hq, Hkv, W):
    assert swa.fwd_path(B, T, Hq, Hkv, 128, W) == "tc_swa"
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=1000 + T + W)
    _full_check(x, W)


@pytest.mark.parametrize("B,T,Hq,Hkv,W", [
    (1, 300, 4, 1, 128),      # 4 heads per kv head: tiles of 32 positions x 4 heads
    (2, 1000, 16, 4, 128),
    (1, 77, 8, 2, 33),
    (1, 300, 4, 1, 1),
    (1, 300, 4, 1, 129),
    (1, 4099, 32, 8, 128),    # many runs per CTA, ragged tail
    (1, 300, 16, 1, 128),     # 16 heads per kv head: two groups of 8 share its keys
    (2, 1000, 64, 4, 128),
    (1, 513, 32, 2, 100),
    (1, 200, 24, 1, 128),     # 24: three groups of 8
    (1, 300, 64, 1, 128),     # 64: eight groups of 8
])
def test_tc_swa_group_sizes(cuda_ok, B, T, Hq, Hkv, W):
    assert swa.fwd_path(B, T, Hq, Hkv, 128, W) == "tc_swa"
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=1100 + T + W + Hq)
    _full_check(x, W)


@pytest.mark.parametrize("B,T,Hq,Hkv,W", [
    (1, 300, 8, 1, 128),      # head dimension 64: 8 heads per tile
    (2, 1000, 16, 4, 128),    # 4 heads per tile
    (1, 700, 32, 2, 100),     # two groups of 8 per kv head
    (1, 77, 8, 1, 1),
    (1, 4099, 64, 8, 129),
])
def test_tc_swa_head_dim_64(cuda_ok, B, T, Hq, Hkv, W):
    assert swa.fwd_path(B, T, Hq, Hkv, 64, W) == "tc_swa"
    x = gen.prefill_inputs(B, T, Hq, Hkv, 64, seed=1200 + T + W + Hq)
    _full_check(x, W)
    o16, l16 = swa.swa_sink_fwd(*(t.cuda() for t in (x.q, x.k, x.v, x.sink)), W,
                                out_dtype=torch.bfloat16)
    o32, l32 = _run(x, W)
    assert torch.equal(o16, o32.to(torch.bfloat16)) and torch.equal(l16, l32)


def test_tc_swa_sink_limits(cuda_ok):
    x = gen.prefill_inputs(1, 200, 8, 1, 128, seed=5)
    # no sink: plain windowed softmax
    x.sink = torch.full((8,), -math.inf)
    _full_check(x, 128)
    # very large sink: output ~ 0, lse = sink
    x.sink = torch.full((8,), 60.0)
    out, lse = _run(x, 128)
    assert out.abs().max().item() < 1e-12
    assert torch.allclose(lse.cpu(), torch.full_like(lse.cpu(), 60.0), atol=1e-4)


def test_tc_swa_without_lse(cuda_ok):
    x = gen.prefill_inputs(1, 100, 8, 1, 128, seed=6)
    q, k, v, s = (t.cuda() for t in (x.q, x.k, x.v, x.sink))
    out, lse = swa.swa_sink_fwd(q, k, v, s, 128, with_lse=False)
    assert lse is None
    ref, _ = swa.swa_sink_fwd(q, k, v, s, 128)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_tc_swa_repeatable(cuda_ok):
    x = gen.prefill_inputs(2, 700, 16, 2, 128, seed=7)
    a, la = _run(x, 128)
    b, lb = _run(x, 128)
    assert torch.equal(a, b) and torch.equal(la, lb)


# ---- masking is exact: huge finite values outside each row's window -------
def test_tc_swa_masked_keys_contribute_nothing(cuda_ok):
    B, T, Hq, Hkv, W = 1, 96, 8, 1, 128
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=8)
    base, lbase = _run(x, 32)
    # tile of positions [48, 64): rows there see keys [i-31, i]; keys in
    # [48-31-17, 48-31) are inside the tile's loaded span but masked for all
    # of its rows -- poison them with huge finite values.
    k, v = x.k.clone(), x.v.clone()
    k[:, 0:17] = 1e30
    v[:, 0:17] = 1e30
    y = gen.PrefillInputs(x.q, k, v, x.sink)
    got, lgot = _run(y, 32)
    assert torch.equal(got[:, 48:64], base[:, 48:64])
    assert torch.equal(lgot[:, :, 48:64], lbase[:, :, 48:64])


def test_tc_swa_does_not_read_outside_tile_span(cuda_ok):
    B, T, Hq, Hkv, W = 1, 512, 8, 1, 128
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=9)
    base, lbase = _run(x, W)
    # tile n = 20 (positions 320..335) loads key blocks 12..20 = keys 192..335
    k, v = x.k.clone(), x.v.clone()
    k[:, :192] = float("nan")
    v[:, :192] = float("nan")
    k[:, 336:] = float("nan")
    v[:, 336:] = float("nan")
    got, lgot = _run(gen.PrefillInputs(x.q, k, v, x.sink), W)
    assert torch.equal(got[:, 320:336], base[:, 320:336])
    assert torch.equal(lgot[:, :, 320:336], lbase[:, :, 320:336])


# ---- general kernel (fp32 path and shapes outside the tensor-core kernel) ---
def test_tiny_fp32_workload(cuda_ok):
    # B=1, T=512, Hq=4, Hkv=1 (GQA 4:1), D=64, W=128, N(0,1), seed 0
    x = gen.prefill_inputs(1, 512, 4, 1, 64, seed=0, dtype=torch.float32)
    assert swa.fwd_path(1, 512, 4, 1, 64, 128, swa.SWA_F32) == "simt"
    _full_check(x, 128, fp32=True)


@pytest.mark.parametrize("B,T,Hq,Hkv,D,W", [
    (2, 77, 4, 2, 128, 9), (1, 130, 6, 3, 64, 300), (1, 64, 2, 2, 64, 1), (1, 1, 4, 1, 64, 128),
])
def test_simt_fp32_shapes(cuda_ok, B, T, Hq, Hkv, D, W):
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=T + W, dtype=torch.float32)
    _full_check(x, W, fp32=True)


@pytest.mark.parametrize("B,T,Hq,Hkv,D,W", [
    (1, 300, 3, 1, 128, 128), (2, 100, 6, 2, 64, 33), (1, 200, 3, 1, 128, 200),
    (1, 150, 12, 1, 128, 128), (1, 180, 12, 1, 64, 180),
])
def test_simt_bf16_shapes(cuda_ok, B, T, Hq, Hkv, D, W):
    assert swa.fwd_path(B, T, Hq, Hkv, D, W) == "simt"
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=T + W + 1)
    _full_check(x, W)


# ---- full-size workloads, every output compared ----------------------------
def test_prefill_full_size_in_full(cuda_ok):
    # B=4, T=8192, Hq=64, Hkv=8, D=128, W=128, N(0,1) -> bf16, sink N(0,1):
    # every element of out and lse against the oracle, one sequence at a time
    B, T, Hq, Hkv, D, W = 4, 8192, 64, 8, 128, 128
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=0, device="cuda")
    out, lse = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    torch.cuda.synchronize()
    for b in range(B):
        o_ref, l_ref = oracle_by_slices(x.q, x.k, x.v, x.sink, W, b, 0, T)
        assert_bf16_close(out[b].cpu().numpy(), o_ref, what=f"sequence {b}")
        assert_lse_close(lse[b].cpu().numpy(), l_ref)


def test_long_context_in_full(cuda_ok):
    # B=1, T=262144, every 97th key x8 (peaky scores), sink U(-4, 4): every
    # element, in slices of 32768 positions (each with its 127-key halo)
    B, T, Hq, Hkv, D, W = 1, 262144, 64, 8, 128, 128
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=5, device="cuda", sink_dist="uniform4",
                           peaky_every=97)
    out, lse = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    torch.cuda.synchronize()
    S = 32768
    for s0 in range(0, T, S):
        o_ref, l_ref = oracle_by_slices(x.q, x.k, x.v, x.sink, W, 0, s0, s0 + S)
        assert_bf16_close(out[0, s0:s0 + S].cpu().numpy(), o_ref, what=f"positions {s0}..")
        assert_lse_close(lse[0, :, s0:s0 + S].cpu().numpy(), l_ref)
    del x, out, lse
    torch.cuda.empty_cache()


# ---- full-size workloads, sampled rows -------------------------------------
def test_prefill_full_size_sampled(cuda_ok):
    # B=4, T=8192, Hq=64, Hkv=8, D=128, W=128, N(0,1) -> bf16, sink N(0,1)
    B, T, Hq, Hkv, D, W = 4, 8192, 64, 8, 128, 128
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=0, device="cuda")
    out, lse = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    rows = sample_rows(B, T, Hq, 48, seed=1, extra_pos=(4095, 4096, 8176))
    o_ref, l_ref = oracle_rows_from_slices(x.q, x.k, x.v, x.sink, W, rows)
    o, l = gather_rows(out, lse, rows)
    assert_bf16_close(o, o_ref)
    assert_lse_close(l, l_ref)


def test_long_context_sampled(cuda_ok):
    # B=1, T=262144, every 97th key x8 (peaky scores), sink U(-4, 4)
    B, T, Hq, Hkv, D, W = 1, 262144, 64, 8, 128, 128
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=5, device="cuda", sink_dist="uniform4",
                           peaky_every=97)
    out, lse = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    rows = sample_rows(B, T, Hq, 24, seed=2, extra_pos=(96, 193, 131071, 262143))
    o_ref, l_ref = oracle_rows_from_slices(x.q, x.k, x.v, x.sink, W, rows)
    o, l = gather_rows(out, lse, rows)
    assert_bf16_close(o, o_ref)
    assert_lse_close(l, l_ref)
    del x, out, lse
    torch.cuda.empty_cache()


def test_hybrid_block_sampled(cuda_ok):
    # one 5:1 block: five W=128 layers, then one global layer (W = T), T=32768
    T, Hq, Hkv, D = 32768, 64, 8, 128
    for layer in range(6):
        W = 128 if layer < 5 else T
        x = gen.prefill_inputs(1, T, Hq, Hkv, D, seed=100 + layer, device="cuda")
        out, lse = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        # window layers: 24 positions; the global layer: the 10 edge positions
        # plus 64 drawn over the whole causal range, every head
        npos = 24 if layer < 5 else 74
        rows = sample_rows(1, T, Hq, npos, seed=layer, extra_pos=(T - 1,))
        o_ref, l_ref = oracle_rows_from_slices(x.q, x.k, x.v, x.sink, W, rows)
        o, l = gather_rows(out, lse, rows)
        assert_bf16_close(o, o_ref, what=f"layer {layer}")
        assert_lse_close(l, l_ref)


def test_no_device_error_recorded(cuda_ok):
    assert swa.device_error() == 0


# ---- bf16 output: the fp32 result rounded, bit for bit -----------------------
@pytest.mark.parametrize("B,T,Hq,Hkv,W", [
    (1, 300, 8, 1, 128), (3, 1000, 16, 2, 128), (1, 700, 8, 1, 700), (2, 513, 16, 2, 300),
    (2, 600, 8, 2, 128), (1, 500, 32, 2, 128), (1, 400, 32, 2, 400),
])
def test_bf16_output_is_rounded_fp32_output(cuda_ok, B, T, Hq, Hkv, W):
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=3000 + T + W, device="cuda")
    o32, l32 = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    o16, l16 = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(l16, l32)
    o_ref, l_ref = oracle.swa_sink_fwd(x.q.cpu(), x.k.cpu(), x.v.cpu(), x.sink.cpu(), W)
    assert_bf16_close(o16.float().cpu().numpy(), o_ref)


def test_bf16_output_needs_a_tensor_core_path(cuda_ok):
    x = gen.prefill_inputs(1, 64, 3, 1, 128, seed=9, device="cuda")
    assert swa.fwd_path(1, 64, 3, 1, 128, 128) == "simt"
    with pytest.raises(swa.SwaError) as e:
        swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, 128, out_dtype=torch.bfloat16)
    assert e.value.status == swa.SWA_EUNSUPPORTED
