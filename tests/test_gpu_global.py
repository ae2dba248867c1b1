"""GPU parity of the online-softmax tensor-core kernel (global layers, W >= T,
and windows wider than the sliding-window kernel covers) against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen
from gpu_helpers import (assert_bf16_close, assert_lse_close, gather_rows,
                         oracle_rows_from_slices, sample_rows)

pytestmark = pytest.mark.gpu


def _run(x, W):
    q, k, v, s = (t.cuda() for t in (x.q, x.k, x.v, x.sink))
    out, lse = swa.swa_sink_fwd(q, k, v, s, W)
    torch.cuda.synchronize()
    return out, lse


def _full_check(x, W):
    out, lse = _run(x, W)
    o_ref, l_ref = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    assert_bf16_close(out.cpu().numpy(), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)
    return out, lse


@pytest.mark.parametrize("B,T,Hq,Hkv,W", [
    (1, 200, 8, 1, 200),      # global, two key blocks, ragged last item
    (1, 1, 8, 1, 130),        # a single position
    (1, 33, 8, 1, 1000),      # one item and one position of the next
    (1, 300, 8, 1, 1000),     # W > T
    (2, 513, 16, 2, 513),     # W = T, crosses 128-key block edges
    (1, 1000, 8, 1, 130),     # just wider than the sliding-window kernel
    (1, 700, 8, 1, 300),      # window start inside a block
    (3, 257, 8, 1, 256),
    (1, 2049, 64, 8, 2049),   # many items per CTA, 17 key blocks
])
def test_tc_global_matches_oracle(cuda_ok, B, T, Hq, Hkv, W):
    assert swa.fwd_path(B, T, Hq, Hkv, 128, W) == "tc_global"
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=2000 + T + W)
    _full_check(x, W)


@pytest.mark.parametrize("B,T,Hq,Hkv,W", [
    (1, 700, 16, 1, 700),     # 16 heads per kv head: two groups of 8 share its keys
    (2, 600, 32, 2, 300),
    (1, 500, 24, 1, 500),     # three groups of 8
    (1, 1100, 64, 1, 1100),   # eight groups: the snake order over (sequence, group) pairs
])
def test_tc_global_group_sizes(cuda_ok, B, T, Hq, Hkv, W):
    assert swa.fwd_path(B, T, Hq, Hkv, 128, W) == "tc_global"
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=2100 + T + W + Hq)
    _full_check(x, W)


def test_tc_global_running_max_moves(cuda_ok):
    # later keys score ever higher, so the running max moves block after block
    # and O is rescaled in tensor memory many times
    B, T, Hq, Hkv, W = 1, 1536, 8, 1, 1536
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=21)
    ramp = torch.linspace(0.2, 3.0, T).view(1, T, 1, 1)
    q = (x.q.float().abs() * 0.0 + 1.0).to(torch.bfloat16)        # all-ones queries
    k = (x.k.float().abs() * ramp).to(torch.bfloat16)             # positive, growing keys
    y = gen.PrefillInputs(q, k, x.v, x.sink)
    _full_check(y, W)


def test_tc_global_peaky_keys(cuda_ok):
    x = gen.prefill_inputs(1, 1200, 16, 2, 128, seed=22, sink_dist="uniform4", peaky_every=97)
    _full_check(x, 1200)


def test_tc_global_sink_limits(cuda_ok):
    x = gen.prefill_inputs(1, 400, 8, 1, 128, seed=23)
    x.sink = torch.full((8,), -math.inf)
    _full_check(x, 400)
    x.sink = torch.full((8,), 60.0)
    out, lse = _run(x, 400)
    assert out.abs().max().item() < 1e-12
    assert torch.allclose(lse.cpu(), torch.full_like(lse.cpu(), 60.0), atol=1e-4)


def test_tc_global_keys_before_window_never_read(cuda_ok):
    # W = 200: positions 512..543 (one item) use key blocks 2..4 only
    x = gen.prefill_inputs(1, 800, 8, 1, 128, seed=24)
    base, lbase = _run(x, 200)
    k, v = x.k.clone(), x.v.clone()
    k[:, :256] = float("nan")
    v[:, :256] = float("nan")
    k[:, 640:] = float("nan")
    v[:, 640:] = float("nan")
    got, lgot = _run(gen.PrefillInputs(x.q, k, v, x.sink), 200)
    assert torch.equal(got[:, 512:544], base[:, 512:544])
    assert torch.equal(lgot[:, :, 512:544], lbase[:, :, 512:544])


def test_tc_global_masked_keys_contribute_nothing(cuda_ok):
    # keys after a row (the causal edge of its last block) and keys before its
    # window start, inside blocks the item loads, hold huge finite values
    x = gen.prefill_inputs(1, 800, 8, 1, 128, seed=25)
    base, lbase = _run(x, 200)
    k, v = x.k.clone(), x.v.clone()
    k[:, 256:312] = 1e30     # before the window of positions 512..543 (first key 313)
    v[:, 256:312] = 1e30
    k[:, 544:640] = 1e30     # after the last position of the item
    v[:, 544:640] = 1e30
    got, lgot = _run(gen.PrefillInputs(x.q, k, v, x.sink), 200)
    assert torch.equal(got[:, 512:544], base[:, 512:544])
    assert torch.equal(lgot[:, :, 512:544], lbase[:, :, 512:544])


def test_tc_global_repeatable(cuda_ok):
    x = gen.prefill_inputs(2, 1100, 16, 2, 128, seed=26)
    a, la = _run(x, 1100)
    b, lb = _run(x, 1100)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_tc_global_wide_window_sampled(cuda_ok):
    # a window of 1024 over 8192 positions, 4 sequences
    B, T, Hq, Hkv, D, W = 4, 8192, 64, 8, 128, 1024
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=27, device="cuda")
    out, lse = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    rows = sample_rows(B, T, Hq, 16, seed=3, extra_pos=(1023, 1024, 8191))
    o_ref, l_ref = oracle_rows_from_slices(x.q, x.k, x.v, x.sink, W, rows)
    o, l = gather_rows(out, lse, rows)
    assert_bf16_close(o, o_ref)
    assert_lse_close(l, l_ref)


@pytest.mark.parametrize("B,T,Hq,Hkv,W", [
    (1, 700, 8, 1, 700),      # global layer, ragged last item
    (2, 513, 16, 2, 300),     # window start inside a block, two groups per kv head
    (1, 1100, 32, 4, 1100),
])
def test_tc_global_head_dim_64(cuda_ok, B, T, Hq, Hkv, W):
    # D = 64: one 128-byte swizzle atom per row, 4 K-steps for S, PV with N = 64
    assert swa.fwd_path(B, T, Hq, Hkv, 64, W) == "tc_global"
    x = gen.prefill_inputs(B, T, Hq, Hkv, 64, seed=2300 + T + W)
    o32, l32 = _full_check(x, W)
    o16, l16 = swa.swa_sink_fwd(*(t.cuda() for t in (x.q, x.k, x.v, x.sink)), W,
                                out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(o16, o32.to(torch.bfloat16)) and torch.equal(l16, l32)


@pytest.mark.parametrize("B,T,Hq,Hkv,D,W", [
    (1, 700, 4, 1, 128, 700),      # 4 heads per kv head: tiles of 32 positions x 4 heads
    (2, 1000, 16, 4, 128, 1000),   # items of 64 positions, the last one ragged
    (1, 900, 8, 2, 128, 300),      # window start inside a block
    (3, 130, 4, 1, 128, 130),
    (1, 1500, 32, 8, 64, 1500),    # head dimension 64
])
def test_tc_global_four_heads_per_kv_head(cuda_ok, B, T, Hq, Hkv, D, W):
    assert swa.fwd_path(B, T, Hq, Hkv, D, W) == "tc_global"
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=2400 + T + W + D)
    o32, l32 = _full_check(x, W)
    o16, l16 = swa.swa_sink_fwd(*(t.cuda() for t in (x.q, x.k, x.v, x.sink)), W,
                                out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(o16, o32.to(torch.bfloat16)) and torch.equal(l16, l32)


@pytest.mark.parametrize("B,T,Hq,Hkv,D,W", [
    (1, 700, 2, 1, 128, 700),      # 2 heads per kv head: tiles of 64 positions x 2 heads
    (2, 600, 8, 4, 64, 128),       # the sliding window on this kernel (its tiles do not fit G = 2)
    (1, 900, 4, 4, 128, 900),      # 1 head per kv head: tiles of 128 positions
    (2, 400, 2, 2, 128, 33),       # 1 head, narrow window
    (1, 1000, 8, 8, 64, 300),
    (1, 1, 2, 2, 128, 128),        # a single position
    (3, 5, 4, 2, 64, 1),           # W = 1: each row sees only its own key
    (1, 257, 2, 1, 128, 257),      # one item (256 positions) and one position of the next
])
def test_tc_global_one_and_two_heads_per_kv_head(cuda_ok, B, T, Hq, Hkv, D, W):
    assert swa.fwd_path(B, T, Hq, Hkv, D, W) == "tc_global"
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=2500 + T + W + D + Hq)
    o32, l32 = _full_check(x, W)
    o16, l16 = swa.swa_sink_fwd(*(t.cuda() for t in (x.q, x.k, x.v, x.sink)), W,
                                out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(o16, o32.to(torch.bfloat16)) and torch.equal(l16, l32)


def test_tc_global_four_heads_per_kv_head_sampled(cuda_ok):
    # B1 T16384 Hq32 Hkv8 D128 global layer: 10 edge positions plus 54 drawn
    # over the causal range, every head
    B, T, Hq, Hkv, D = 1, 16384, 32, 8, 128
    assert swa.fwd_path(B, T, Hq, Hkv, D, T) == "tc_global"
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=2450, device="cuda")
    out, lse = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, T)
    torch.cuda.synchronize()
    rows = sample_rows(B, T, Hq, 64, seed=44)
    o_ref, l_ref = oracle_rows_from_slices(x.q, x.k, x.v, x.sink, T, rows)
    o, l = gather_rows(out, lse, rows)
    assert_bf16_close(o, o_ref)
    assert_lse_close(l, l_ref)


def test_tc_global_no_device_error(cuda_ok):
    assert swa.device_error() == 0
