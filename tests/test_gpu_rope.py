"""GPU rotary embedding and the fused rotate-and-append step against the
fp64 oracle.  Outputs are in the input dtype: bf16 results may differ from the
correctly rounded fp64 value by one rounding (relative 2^-8)."""
import numpy as np
import pytest
import torch

import oracle
import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen
from gpu_helpers import assert_bf16_close, assert_lse_close

pytestmark = pytest.mark.gpu

THETA = 10000.0


def _close_to_rounding(got, ref, dtype):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if dtype == torch.bfloat16:
        tol = 2.0 ** -8 * np.abs(ref) + 1e-6
    else:
        tol = 1e-5 * np.abs(ref).max() + 1e-7
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} elements off; worst {np.abs(got - ref).max():.3e}"


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D,rot", [(128, 128), (128, 64), (64, 64)])
def test_rope_matches_oracle(cuda_ok, dt, D, rot):
    g = torch.Generator().manual_seed(7 + D + rot)
    x = torch.randn(3, 200, 8, D, generator=g).to(dt)
    pos0 = torch.tensor([0, 131000, 262144 - 200], dtype=torch.int64)
    xd = x.cuda()
    swa.swa_rope(xd, pos0.cuda(), rot, THETA)
    torch.cuda.synchronize()
    ref = oracle.rope(x, pos0, rot, THETA)
    _close_to_rounding(xd.cpu().double().numpy(), ref, dt)
    # dimensions past rot_dim are untouched, bit for bit
    assert torch.equal(xd[..., rot:].cpu(), x[..., rot:])


def test_rope_append_matches_oracle(cuda_ok):
    B, Hq, Hkv, D, W = 6, 64, 8, 128, 128
    d = gen.decode_inputs(B, Hq, Hkv, D, W, seed=71, pos_lo=0, pos_hi=262144)
    d.pos[0] = 0
    d.pos[1] = W - 1
    d.pos[2] = -3            # negative: nothing written
    g = torch.Generator().manual_seed(72)
    k = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    kr, vr, qd = d.k_ring.cuda(), d.v_ring.cuda(), d.q.cuda()
    q_out = torch.full_like(qd, 7.0)
    swa.swa_rope_append(qd, k.cuda(), v.cuda(), kr, vr, d.pos.cuda(), 128, THETA, q_out=q_out)
    torch.cuda.synchronize()
    pos_ok = d.pos.clamp(min=0)
    q_ref = oracle.rope(d.q.unsqueeze(1), pos_ok, 128, THETA)[:, 0]
    k_ref = oracle.rope(k.unsqueeze(1), pos_ok, 128, THETA)[:, 0]
    kr_h, vr_h, qo_h = kr.cpu(), vr.cpu(), q_out.cpu()
    for b in range(B):
        p = int(d.pos[b])
        if p < 0:
            assert torch.equal(kr_h[b], d.k_ring[b]) and torch.equal(vr_h[b], d.v_ring[b])
            assert torch.all(qo_h[b] == 7.0)
            continue
        s = p % W
        _close_to_rounding(qo_h[b].double().numpy(), q_ref[b], torch.bfloat16)
        _close_to_rounding(kr_h[b, :, s].double().numpy(), k_ref[b], torch.bfloat16)
        assert torch.equal(vr_h[b, :, s], v[b])
        others = [t for t in range(W) if t != s]
        assert torch.equal(kr_h[b][:, others], d.k_ring[b][:, others])
        assert torch.equal(vr_h[b][:, others], d.v_ring[b][:, others])


def test_rotate_append_decode_equals_rotated_prefill(cuda_ok):
    # a history of unrotated q, k: rotating it all and running the prefill, or
    # feeding it token by token through rope_append + decode, give one result
    B, T, Hq, Hkv, D, W = 2, 300, 16, 2, 128, 128
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=73)
    pos0 = torch.zeros(B, dtype=torch.int64)
    qr = oracle.rope(x.q, pos0, D, THETA)
    kr_ = oracle.rope(x.k, pos0, D, THETA)
    # oracle: rotated (then bf16-rounded, as the kernels store them) history
    q16 = torch.from_numpy(qr).to(torch.bfloat16)
    k16 = torch.from_numpy(kr_).to(torch.bfloat16)
    o_ref, l_ref = oracle.swa_sink_fwd(q16, k16, x.v, x.sink, W)
    kring = torch.zeros(B, Hkv, W, D, dtype=torch.bfloat16, device="cuda")
    vring = torch.zeros_like(kring)
    qd, kd, vd, sd = (t.cuda() for t in (x.q, x.k, x.v, x.sink))
    worst, lworst = 0.0, 0.0
    for t in range(T):
        pos = torch.full((B,), t, dtype=torch.int64, device="cuda")
        q_t = swa.swa_rope_append(qd[:, t].contiguous(), kd[:, t].contiguous(),
                                  vd[:, t].contiguous(), kring, vring, pos, D, THETA)
        o, l = swa.swa_sink_decode(q_t, kring, vring, pos, sd)
        if t % 37 == 0 or t == T - 1:
            torch.cuda.synchronize()
            worst = max(worst, np.abs(o.cpu().double().numpy() - o_ref[:, t]).max())
            lworst = max(lworst, np.abs(l.cpu().double().numpy() - l_ref[:, :, t]).max())
    assert worst <= 2e-2, worst
    assert lworst <= 1e-3, lworst
    assert swa.device_error() == 0


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,T,H", [(3, 5, 1), (4, 3, 2), (2, 9, 3)])
def test_rope_groups_of_tokens_across_sequences(cuda_ok, dt, B, T, H):
    # few heads per token: a block takes up to 8 tokens at a time, which here
    # span several sequences with unrelated start positions
    D, rot = 64, 64
    g = torch.Generator().manual_seed(90 + B * T * H)
    x = torch.randn(B, T, H, D, generator=g).to(dt)
    pos0 = torch.tensor([7, 262140, 0, 99999][:B], dtype=torch.int64)
    xd = x.cuda()
    swa.swa_rope(xd, pos0.cuda(), rot, THETA)
    torch.cuda.synchronize()
    _close_to_rounding(xd.cpu().double().numpy(), oracle.rope(x, pos0, rot, THETA), dt)
    assert swa.device_error() == 0
