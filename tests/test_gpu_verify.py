"""GPU parity of the multi-token verify (drafted tokens checked in one pass
against the ring) with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen
from gpu_helpers import assert_bf16_close, assert_f32_close, assert_lse_close

pytestmark = pytest.mark.gpu


def _verify(x):
    args = [t.cuda() for t in (x.q, x.k_new, x.v_new, x.k_ring, x.v_ring, x.pos, x.sink)]
    out, lse = swa.swa_sink_verify(*args)
    torch.cuda.synchronize()
    return out.cpu().double().numpy(), lse.cpu().double().numpy()


def _oracle(x):
    return oracle.swa_sink_verify(x.q, x.k_new, x.v_new, x.k_ring, x.v_ring, x.pos, x.sink)


def _check(x, fp32=False):
    o, l = _verify(x)
    o_ref, l_ref = _oracle(x)
    if fp32:
        assert_f32_close(o, o_ref)
        assert_f32_close(l, l_ref, what="lse")
    else:
        assert_bf16_close(o, o_ref)
        assert_lse_close(l, l_ref)


def test_verify_mtp_workload(cuda_ok):
    # 256 sequences, 4 drafted tokens each (the token plus three drafts),
    # Hq=64, Hkv=8, D=128, W=128 ring, positions U[128, 262144)
    x = gen.verify_inputs(256, 4, 64, 8, 128, 128, seed=0)
    _check(x)


@pytest.mark.parametrize("B,L,Hq,Hkv,D,W,dt", [
    (3, 1, 8, 1, 128, 128, torch.bfloat16),
    (3, 2, 16, 2, 128, 128, torch.bfloat16),
    (5, 3, 8, 1, 128, 128, torch.bfloat16),
    (2, 4, 64, 8, 128, 128, torch.bfloat16),
    (2, 7, 8, 1, 128, 128, torch.bfloat16),
    (3, 4, 4, 2, 64, 33, torch.bfloat16),
    (2, 5, 8, 8, 64, 4, torch.bfloat16),       # more drafts than the window
    (3, 3, 8, 1, 128, 128, torch.float32),
    (2, 2, 4, 4, 64, 300, torch.float32),
])
def test_verify_shapes(cuda_ok, B, L, Hq, Hkv, D, W, dt):
    x = gen.verify_inputs(B, L, Hq, Hkv, D, W, seed=B + L + W, dtype=dt, pos_lo=0, pos_hi=4 * W)
    _check(x, fp32=dt == torch.float32)


@pytest.mark.parametrize("B,L,pos_hi", [(37, 5, 600), (29, 6, 300), (41, 8, 2000), (9, 8, 9)])
def test_verify_tc_up_to_eight_drafts(cuda_ok, B, L, pos_hi):
    # 5 to 8 drafted tokens on the tensor cores (64 query rows per group, two
    # softmax warps per warpgroup), full and partial rings with NaN in the
    # empty slots, positions where every window still starts at 0
    assert swa.verify_path(B, L, 64, 8, 128, 128) == "tc_verify"
    x = gen.verify_inputs(B, L, 64, 8, 128, 128, seed=B + L, pos_lo=0, pos_hi=pos_hi)
    for b in range(B):
        p = int(x.pos[b])
        if p < 128:
            x.k_ring[b, :, p:] = float("nan")
            x.v_ring[b, :, p:] = float("nan")
    _check(x)
    assert swa.device_error() == 0


@pytest.mark.parametrize("B,L", [(33, 4), (21, 8), (7, 1)])
def test_verify_tc_head_dim_64(cuda_ok, B, L):
    assert swa.verify_path(B, L, 64, 8, 64, 128) == "tc_verify"
    x = gen.verify_inputs(B, L, 64, 8, 64, 128, seed=B + L + 64, pos_lo=0, pos_hi=700)
    for b in range(B):
        p = int(x.pos[b])
        if p < 128:
            x.k_ring[b, :, p:] = float("nan")
            x.v_ring[b, :, p:] = float("nan")
    _check(x)
    assert swa.device_error() == 0


@pytest.mark.parametrize("B,L,Hq,Hkv,D", [(23, 4, 64, 4, 128), (17, 8, 96, 4, 128),
                                          (30, 3, 32, 1, 64), (151, 2, 64, 4, 128)])
def test_verify_tc_sibling_groups(cuda_ok, B, L, Hq, Hkv, D):
    # 16, 24 and 32 query heads per kv head: sibling groups of 8 on the same
    # rings and drafted keys; B = 151 with 4 kv heads and 2 siblings gives
    # CTAs 8 or 9 groups, sibling pairs split across rounds
    assert swa.verify_path(B, L, Hq, Hkv, D, 128) == "tc_verify"
    x = gen.verify_inputs(B, L, Hq, Hkv, D, 128, seed=B + L + Hq, pos_lo=0, pos_hi=700)
    for b in range(B):
        p = int(x.pos[b])
        if p < 128:
            x.k_ring[b, :, p:] = float("nan")
            x.v_ring[b, :, p:] = float("nan")
    _check(x)
    assert swa.device_error() == 0


@pytest.mark.parametrize("B,L,Hq,Hkv,D", [(19, 4, 16, 4, 128), (13, 8, 32, 8, 64),
                                          (21, 3, 8, 4, 128), (9, 8, 4, 4, 128),
                                          (150, 5, 8, 2, 128)])
def test_verify_tc_small_groups(cuda_ok, B, L, Hq, Hkv, D):
    # 4, 2 and 1 query heads per kv head: rows r = G j + h of one 32-row
    # group; B = 150 with 2 kv heads gives CTAs 2 or 3 groups
    assert swa.verify_path(B, L, Hq, Hkv, D, 128) == "tc_verify"
    x = gen.verify_inputs(B, L, Hq, Hkv, D, 128, seed=B + L + Hq + 7, pos_lo=0, pos_hi=700)
    for b in range(B):
        p = int(x.pos[b])
        if p < 128:
            x.k_ring[b, :, p:] = float("nan")
            x.v_ring[b, :, p:] = float("nan")
    _check(x)
    assert swa.device_error() == 0


def test_verify_eight_drafts_equal_prefill_rows(cuda_ok):
    B, T, Hq, Hkv, D, W, L = 2, 600, 16, 2, 128, 128, 8
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=64, device="cuda")
    out_pre, lse_pre = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    pos = torch.tensor([5, 401], dtype=torch.int64)
    kr, vr = gen.ring_from_history(x.k.cpu(), x.v.cpu(), pos - 1, W)
    idx = [torch.arange(int(p), int(p) + L) for p in pos]
    qn = torch.stack([x.q[b, idx[b]] for b in range(B)]).contiguous()
    kn = torch.stack([x.k[b, idx[b]] for b in range(B)]).contiguous()
    vn = torch.stack([x.v[b, idx[b]] for b in range(B)]).contiguous()
    assert swa.verify_path(B, L, Hq, Hkv, D, W) == "tc_verify"
    o, l = swa.swa_sink_verify(qn, kn, vn, kr.cuda(), vr.cuda(), pos.cuda(), x.sink)
    torch.cuda.synchronize()
    for b in range(B):
        p = int(pos[b])
        assert (o[b] - out_pre[b, p:p + L]).abs().max().item() < 2e-2
        assert (l[b] - lse_pre[b, :, p:p + L]).abs().max().item() < 1e-3


def test_verify_equals_prefill_rows_on_gpu(cuda_ok):
    # drafts checked against a ring laid from the history equal the GPU prefill
    B, T, Hq, Hkv, D, W, L = 3, 400, 16, 2, 128, 128, 4
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=61, device="cuda")
    out_pre, lse_pre = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    pos = torch.tensor([0, 100, 333], dtype=torch.int64)
    kr, vr = gen.ring_from_history(x.k.cpu(), x.v.cpu(), pos - 1, W)
    idx = [torch.arange(int(p), int(p) + L) for p in pos]
    qn = torch.stack([x.q[b, idx[b]] for b in range(B)]).contiguous()
    kn = torch.stack([x.k[b, idx[b]] for b in range(B)]).contiguous()
    vn = torch.stack([x.v[b, idx[b]] for b in range(B)]).contiguous()
    o, l = swa.swa_sink_verify(qn, kn, vn, kr.cuda(), vr.cuda(), pos.cuda(), x.sink)
    torch.cuda.synchronize()
    for b in range(B):
        p = int(pos[b])
        assert (o[b] - out_pre[b, p:p + L]).abs().max().item() < 2e-2
        assert (l[b] - lse_pre[b, :, p:p + L]).abs().max().item() < 1e-3


def test_verify_empty_slots_ignored_even_if_nan(cuda_ok):
    W = 128
    x = gen.verify_inputs(6, 3, 64, 8, 128, W, seed=62, pos_lo=0, pos_hi=W)
    ref = _verify(x)
    for b in range(6):
        p = int(x.pos[b])
        x.k_ring[b, :, p:] = float("nan")     # slots s >= pos hold negative positions
        x.v_ring[b, :, p:] = float("nan")
    got = _verify(x)
    assert np.all(np.isfinite(got[0])) and np.all(np.isfinite(got[1]))
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    o_ref, l_ref = _oracle(x)
    assert_bf16_close(got[0], o_ref)
    assert_lse_close(got[1], l_ref)


def test_verify_negative_position_is_empty(cuda_ok):
    x = gen.verify_inputs(3, 2, 16, 2, 128, 128, seed=63, pos_lo=0, pos_hi=500)
    x.pos[1] = -1
    o, l = _verify(x)
    assert np.all(o[1] == 0.0)
    assert np.allclose(l[1], x.sink.double().numpy()[:, None], atol=1e-6)


def test_verify_no_device_error(cuda_ok):
    assert swa.device_error() == 0
