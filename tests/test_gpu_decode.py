"""GPU decode and ring-append parity against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen
from gpu_helpers import assert_bf16_close, assert_f32_close, assert_lse_close

pytestmark = pytest.mark.gpu


def _decode(x):
    args = [t.cuda() for t in (x.q, x.k_ring, x.v_ring, x.pos, x.sink)]
    out, lse = swa.swa_sink_decode(*args)
    torch.cuda.synchronize()
    return out.cpu().double().numpy(), lse.cpu().double().numpy()


def test_decode_full_size_workload(cuda_ok):
    # 256 sequences at positions U[128, 262144), Hq=64, Hkv=8, D=128, W=128 ring
    x = gen.decode_inputs(256, 64, 8, 128, 128, seed=0)
    o, l = _decode(x)
    o_ref, l_ref = oracle.swa_sink_decode(x.q, x.k_ring, x.v_ring, x.pos, x.sink)
    assert_bf16_close(o, o_ref)
    assert_lse_close(l, l_ref)


@pytest.mark.parametrize("B,Hq,Hkv", [(37, 64, 16), (29, 64, 4), (11, 8, 4), (13, 4, 4),
                                       (300, 16, 1), (20, 96, 4), (33, 64, 2), (77, 128, 4)])
def test_decode_tc_group_sizes(cuda_ok, B, Hq, Hkv):
    # the tensor-core decode for 4, 16, 2 and 1 query heads per kv head (the
    # 16 MMA columns hold the group's heads, the rest padding), and for 24, 32
    # and 32 again as sibling groups of 8 on the same rings; partial and full
    # rings, one and several groups per sequence
    assert swa.decode_path(B, Hq, Hkv, 128, 128) == "tc_decode"
    x = gen.decode_inputs(B, Hq, Hkv, 128, 128, seed=B + Hq, pos_lo=0, pos_hi=600)
    for b in range(B):
        p = int(x.pos[b])
        if p < 127:   # empty slots may hold anything
            x.k_ring[b, :, p + 1:] = float("nan")
            x.v_ring[b, :, p + 1:] = float("nan")
    o, l = _decode(x)
    o_ref, l_ref = oracle.swa_sink_decode(x.q, x.k_ring, x.v_ring, x.pos, x.sink)
    assert_bf16_close(o, o_ref)
    assert_lse_close(l, l_ref)
    assert swa.device_error() == 0


@pytest.mark.parametrize("B,Hq,Hkv", [(37, 64, 8), (29, 64, 4), (13, 8, 8), (50, 16, 4), (41, 16, 8),
                                      (300, 64, 8)])   # 16 or 17 groups per CTA: three warpgroups in turn
def test_decode_tc_head_dim_64(cuda_ok, B, Hq, Hkv):
    # head dimension 64 on the tensor cores, partial rings with NaN in the empty slots
    assert swa.decode_path(B, Hq, Hkv, 64, 128) == "tc_decode"
    x = gen.decode_inputs(B, Hq, Hkv, 64, 128, seed=B + Hq + 64, pos_lo=0, pos_hi=600)
    for b in range(B):
        p = int(x.pos[b])
        if p < 127:
            x.k_ring[b, :, p + 1:] = float("nan")
            x.v_ring[b, :, p + 1:] = float("nan")
    o, l = _decode(x)
    o_ref, l_ref = oracle.swa_sink_decode(x.q, x.k_ring, x.v_ring, x.pos, x.sink)
    assert_bf16_close(o, o_ref)
    assert_lse_close(l, l_ref)
    assert swa.device_error() == 0


@pytest.mark.parametrize("B,Hq,Hkv,D,W,dt", [
    (3, 8, 1, 128, 128, torch.bfloat16), (5, 16, 1, 64, 64, torch.bfloat16),
    (4, 4, 2, 128, 33, torch.bfloat16), (2, 16, 16, 64, 7, torch.bfloat16),
    (3, 8, 1, 128, 128, torch.float32), (2, 4, 4, 64, 300, torch.float32),
    (3, 24, 8, 128, 64, torch.bfloat16),    # 3 heads per kv head: three 1-head sibling CTAs
    (2, 48, 2, 64, 33, torch.bfloat16),     # 24: three 8-head siblings
    (2, 12, 1, 128, 100, torch.float32),    # 12: three 4-head siblings
])
def test_decode_shapes(cuda_ok, B, Hq, Hkv, D, W, dt):
    x = gen.decode_inputs(B, Hq, Hkv, D, W, seed=B + W, dtype=dt, pos_lo=0, pos_hi=4 * W)
    o, l = _decode(x)
    o_ref, l_ref = oracle.swa_sink_decode(x.q, x.k_ring, x.v_ring, x.pos, x.sink)
    if dt == torch.float32:
        assert_f32_close(o, o_ref)
        assert_f32_close(l, l_ref, what="lse")
    else:
        assert_bf16_close(o, o_ref)
        assert_lse_close(l, l_ref)


def test_decode_empty_slots_ignored_even_if_nan(cuda_ok):
    W = 128
    x = gen.decode_inputs(6, 64, 8, 128, W, seed=3, pos_lo=0, pos_hi=W - 1)
    ref = _decode(x)
    for b in range(6):
        p = int(x.pos[b])
        x.k_ring[b, :, p + 1:] = float("nan")
        x.v_ring[b, :, p + 1:] = float("nan")
    got = _decode(x)
    assert np.all(np.isfinite(got[0])) and np.all(np.isfinite(got[1]))
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    o_ref, l_ref = oracle.swa_sink_decode(x.q, x.k_ring, x.v_ring, x.pos, x.sink)
    assert_bf16_close(got[0], o_ref)
    assert_lse_close(got[1], l_ref)


def test_ring_append_bit_exact(cuda_ok):
    B, Hkv, W, D = 7, 8, 128, 128
    g = torch.Generator().manual_seed(4)
    kr = torch.randn(B, Hkv, W, D, generator=g).to(torch.bfloat16)
    vr = torch.randn(B, Hkv, W, D, generator=g).to(torch.bfloat16)
    kn = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    pos = torch.tensor([0, 1, 127, 128, 129, 262143, -1], dtype=torch.int64)
    kr_d, vr_d = kr.cuda(), vr.cuda()
    swa.swa_ring_append(kn.cuda(), vn.cuda(), kr_d, vr_d, pos.cuda())
    torch.cuda.synchronize()
    for b in range(B):
        p = int(pos[b])
        if p >= 0:
            kr[b, :, p % W] = kn[b]
            vr[b, :, p % W] = vn[b]
    assert torch.equal(kr_d.cpu(), kr) and torch.equal(vr_d.cpu(), vr)


def test_decode_after_appends_equals_prefill_row(cuda_ok):
    # feed a history token by token through the ring; decode at every step
    # must match the prefill row at that position (positions only grow)
    B, T, Hq, Hkv, D, W = 2, 200, 16, 2, 128, 128
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=11, device="cuda")
    out_pre, lse_pre = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    kr = torch.full((B, Hkv, W, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vr = torch.full_like(kr, float("nan"))
    worst = 0.0
    for t in range(T):
        pos = torch.full((B,), t, dtype=torch.int64, device="cuda")
        swa.swa_ring_append(x.k[:, t].contiguous(), x.v[:, t].contiguous(), kr, vr, pos)
        o, l = swa.swa_sink_decode(x.q[:, t].contiguous(), kr, vr, pos, x.sink)
        worst = max(worst, (o - out_pre[:, t]).abs().max().item())
        assert torch.isfinite(o).all()
        assert (l - lse_pre[:, :, t]).abs().max().item() < 1e-3
    torch.cuda.synchronize()
    assert worst < 2e-2
    # and the last step against the oracle
    o_ref, l_ref = oracle.swa_sink_fwd_rows(x.q.cpu(), x.k.cpu(), x.v.cpu(), x.sink.cpu(), W,
                                            [[b, h, T - 1] for b in range(B) for h in range(Hq)])
    assert_bf16_close(o.cpu().double().numpy().reshape(-1, D), o_ref)


def test_tc_decode_selected_for_the_workload_shape(cuda_ok):
    assert swa.decode_path(256, 64, 8, 128, 128) == "tc_decode"
    assert swa.decode_path(3, 8, 1, 128, 128) == "tc_decode"
    assert swa.decode_path(3, 8, 1, 128, 64) == "simt_decode"


def test_tc_decode_negative_position_is_empty(cuda_ok):
    # a negative position leaves every slot empty: out = 0, lse = sink
    x = gen.decode_inputs(3, 16, 2, 128, 128, seed=9, pos_lo=0, pos_hi=500)
    x.pos[1] = -1
    o, l = _decode(x)
    assert np.all(o[1] == 0.0)
    assert np.allclose(l[1], x.sink.double().numpy(), atol=1e-6)
    keep = [0, 2]
    o_ref, l_ref = oracle.swa_sink_decode(x.q[keep], x.k_ring[keep], x.v_ring[keep],
                                          x.pos[keep], x.sink)
    assert_bf16_close(o[keep], o_ref)
    assert_lse_close(l[keep], l_ref)


def test_tc_decode_uneven_groups_per_cta(cuda_ok):
    # more groups than SMs and not a multiple of them: CTAs take 2 or 3 groups
    x = gen.decode_inputs(37, 64, 8, 128, 128, seed=10)
    o, l = _decode(x)
    o_ref, l_ref = oracle.swa_sink_decode(x.q, x.k_ring, x.v_ring, x.pos, x.sink)
    assert_bf16_close(o, o_ref)
    assert_lse_close(l, l_ref)


def test_decode_no_device_error(cuda_ok):
    assert swa.device_error() == 0
