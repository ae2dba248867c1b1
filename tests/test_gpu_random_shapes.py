"""Seeded random shapes through every path selection: prefill (each kernel the
sizes pick), decode, verify and the host-memory prefill, in bf16 and fp32, each
compared element by element with the fp64 oracle (the host-memory prefill bit
for bit with the device call); rotary embedding, the fused rotate-and-append
step and the plain ring append likewise.  The draws mix group sizes the tensor-core kernels take
with ones they do not, windows on both sides of the sliding-window kernel's
limit, ragged lengths and partial rings."""
import numpy as np
import pytest
import torch

import oracle
import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen
from gpu_helpers import assert_bf16_close, assert_f32_close, assert_lse_close

pytestmark = pytest.mark.gpu

GROUPS = (1, 2, 3, 4, 8, 16, 24)


def _prefill_case(seed):
    g = np.random.default_rng(seed)
    G = int(g.choice(GROUPS))
    Hkv = int(g.integers(1, 4))
    D = int(g.choice((64, 128)))
    T = int(g.integers(1, 700))
    B = int(g.integers(1, 4))
    W = int(g.choice((1, 17, 128, 129, 130, 300, T, T + 5)))
    fp32 = bool(g.random() < 0.25)
    return B, T, G * Hkv, Hkv, D, max(W, 1), fp32


@pytest.mark.parametrize("seed", range(32))
def test_random_prefill_shape(cuda_ok, seed):
    B, T, Hq, Hkv, D, W, fp32 = _prefill_case(seed)
    dt = torch.float32 if fp32 else torch.bfloat16
    path = swa.fwd_path(B, T, Hq, Hkv, D, W, swa.SWA_F32 if fp32 else swa.SWA_BF16)
    assert path in ("tc_swa", "tc_global", "simt")
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7000 + seed, dtype=dt)
    out, lse = swa.swa_sink_fwd(*(t.cuda() for t in (x.q, x.k, x.v, x.sink)), W)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    if fp32:
        assert_f32_close(out.cpu().double().numpy(), o_ref, what=f"out ({path})")
        assert_f32_close(lse.cpu().double().numpy(), l_ref, what=f"lse ({path})")
    else:
        assert_bf16_close(out.cpu().numpy(), o_ref, what=f"out ({path})")
        assert_lse_close(lse.cpu().numpy(), l_ref)
    assert swa.device_error() == 0


def _ring_case(seed):
    g = np.random.default_rng(seed)
    G = int(g.choice(GROUPS))
    Hkv = int(g.integers(1, 4))
    D = int(g.choice((64, 128)))
    B = int(g.integers(1, 60))
    W = int(g.choice((128, 128, 64, 33)))
    L = int(g.integers(1, 9))
    fp32 = bool(g.random() < 0.25)
    return B, G * Hkv, Hkv, D, W, L, fp32


def _close(out, lse, o_ref, l_ref, fp32, path):
    o, l = out.cpu().double().numpy(), lse.cpu().double().numpy()
    if fp32:
        assert_f32_close(o, o_ref, what=f"out ({path})")
        assert_f32_close(l, l_ref, what=f"lse ({path})")
    else:
        assert_bf16_close(o, o_ref, what=f"out ({path})")
        assert_lse_close(l, l_ref)


def _poison_empty_slots(x, ring_pos):
    # slots past the newest ring position of a young sequence are empty and
    # may hold anything
    W = x.k_ring.shape[2]
    for b in range(x.k_ring.shape[0]):
        p = int(ring_pos[b])          # -1: an empty ring
        if p < W - 1:
            x.k_ring[b, :, p + 1:] = float("nan")
            x.v_ring[b, :, p + 1:] = float("nan")


@pytest.mark.parametrize("seed", range(24))
def test_random_decode_shape(cuda_ok, seed):
    B, Hq, Hkv, D, W, _, fp32 = _ring_case(seed)
    dt = torch.float32 if fp32 else torch.bfloat16
    x = gen.decode_inputs(B, Hq, Hkv, D, W, seed=7100 + seed, dtype=dt, pos_lo=0, pos_hi=4 * W)
    _poison_empty_slots(x, x.pos)
    out, lse = swa.swa_sink_decode(*(t.cuda() for t in (x.q, x.k_ring, x.v_ring, x.pos, x.sink)))
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.swa_sink_decode(x.q, x.k_ring, x.v_ring, x.pos, x.sink)
    path = swa.decode_path(B, Hq, Hkv, D, W, swa.SWA_F32 if fp32 else swa.SWA_BF16)
    _close(out, lse, o_ref, l_ref, fp32, path)
    assert swa.device_error() == 0


@pytest.mark.parametrize("seed", range(24))
def test_random_verify_shape(cuda_ok, seed):
    B, Hq, Hkv, D, W, L, fp32 = _ring_case(seed + 100)
    dt = torch.float32 if fp32 else torch.bfloat16
    x = gen.verify_inputs(B, L, Hq, Hkv, D, W, seed=7200 + seed, dtype=dt, pos_lo=0, pos_hi=4 * W)
    _poison_empty_slots(x, x.pos - 1)   # the ring holds the tokens before pos
    args = (x.q, x.k_new, x.v_new, x.k_ring, x.v_ring, x.pos, x.sink)
    out, lse = swa.swa_sink_verify(*(t.cuda() for t in args))
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.swa_sink_verify(*args)
    path = swa.verify_path(B, L, Hq, Hkv, D, W, swa.SWA_F32 if fp32 else swa.SWA_BF16)
    _close(out, lse, o_ref, l_ref, fp32, path)
    assert swa.device_error() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_host_prefill_shape(cuda_ok, seed):
    B, T, Hq, Hkv, D, W, fp32 = _prefill_case(seed + 500)
    dt = torch.float32 if fp32 else torch.bfloat16
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7300 + seed, dtype=dt)
    qh, kh, vh = (t.pin_memory() for t in (x.q, x.k, x.v))
    out_h, lse_h, _ = swa.swa_sink_fwd_host(qh, kh, vh, x.sink.cuda(), W)
    out_d, lse_d = swa.swa_sink_fwd(*(t.cuda() for t in (x.q, x.k, x.v, x.sink)), W)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    assert swa.device_error() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_high_sparse_pipeline(cuda_ok, seed):
    # block scores of a global layer, top-k selection on them, and the sparse
    # layer on the selection, each step against the oracle on the GPU's own
    # input to that step
    g = np.random.default_rng(7400 + seed)
    B, Hkv = int(g.integers(1, 3)), int(g.integers(1, 3))
    Hq, D = 8 * Hkv, int(g.choice((64, 128)))
    T = int(g.integers(1, 1500))
    QB, topk = int(g.choice((32, 64, 128))), int(g.integers(1, 9))
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7400 + seed)
    q, k, v, s = (t.cuda() for t in (x.q, x.k, x.v, x.sink))
    _, _, bm = swa.swa_sink_fwd_scores(q, k, v, s, T)
    idx = swa.swa_topk_blocks(bm, T, QB, topk)
    out, lse = swa.swa_sink_sparse_fwd(q, k, v, s, idx, QB)
    torch.cuda.synchronize()
    got = bm.cpu().double().numpy()
    ref = oracle.block_max(x.q, x.k, T)
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    fin = np.isfinite(ref)
    if fin.any():
        assert np.abs(got[fin] - ref[fin]).max() <= 1e-3
    assert np.array_equal(idx.cpu().numpy(), oracle.topk_blocks(bm.cpu().numpy(), T, QB, topk))
    o_ref, l_ref = oracle.sparse_fwd(x.q, x.k, x.v, x.sink, idx.cpu().numpy(), QB)
    assert_bf16_close(out.cpu().numpy(), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)
    assert swa.device_error() == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_prefill_long(cuda_ok, seed):
    # longer sequences: many tiles and items per CTA, every element compared
    g = np.random.default_rng(7500 + seed)
    G = int(g.choice((1, 2, 4, 8, 16)))
    Hkv = 1 if G == 16 else int(g.integers(1, 3))
    D = int(g.choice((64, 128)))
    T = int(g.integers(1500, 5000))
    B = int(g.integers(1, 3))
    W = int(g.choice((128, 1000, T)))
    Hq = G * Hkv
    path = swa.fwd_path(B, T, Hq, Hkv, D, W)
    assert path in ("tc_swa", "tc_global")
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7500 + seed)
    out, lse = swa.swa_sink_fwd(*(t.cuda() for t in (x.q, x.k, x.v, x.sink)), W)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    assert_bf16_close(out.cpu().numpy(), o_ref, what=f"out ({path})")
    assert_lse_close(lse.cpu().numpy(), l_ref)
    assert swa.device_error() == 0


def _rope_close(got, ref, fp32):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    # bf16: one rounding of the result (relative 2^-8); fp32: normwise 1e-5
    tol = (1e-5 * np.abs(ref).max() + 1e-7) if fp32 else (2.0 ** -8 * np.abs(ref) + 1e-6)
    assert (np.abs(got - ref) <= tol).all(), np.abs(got - ref).max()


def _rope_case(g):
    D = int(g.choice((64, 128)))
    rot = int(g.choice((2, 16, D // 2, D - 2, D)))
    theta = float(g.choice((100.0, 1e4, 5e5)))
    fp32 = bool(g.random() < 0.5)
    return D, rot, theta, fp32


@pytest.mark.parametrize("seed", range(12))
def test_random_rope_shape(cuda_ok, seed):
    g = np.random.default_rng(7600 + seed)
    D, rot, theta, fp32 = _rope_case(g)
    B, T, H = int(g.integers(1, 4)), int(g.integers(1, 400)), int(g.integers(1, 20))
    dt = torch.float32 if fp32 else torch.bfloat16
    tg = torch.Generator().manual_seed(7600 + seed)
    x = torch.randn(B, T, H, D, generator=tg).to(dt)
    pos0 = torch.from_numpy(g.integers(0, 1 << 20, size=B)).to(torch.int64)
    xd = x.cuda()
    swa.swa_rope(xd, pos0.cuda(), rot, theta)
    torch.cuda.synchronize()
    _rope_close(xd.cpu().double().numpy(), oracle.rope(x, pos0, rot, theta), fp32)
    assert torch.equal(xd[..., rot:].cpu(), x[..., rot:])
    assert swa.device_error() == 0


@pytest.mark.parametrize("seed", range(12))
def test_random_rope_append_shape(cuda_ok, seed):
    g = np.random.default_rng(7700 + seed)
    D, rot, theta, fp32 = _rope_case(g)
    B, Hkv = int(g.integers(1, 40)), int(g.integers(1, 4))
    Hq, W = Hkv * int(g.choice(GROUPS)), int(g.choice((1, 33, 128, 200)))
    dt = torch.float32 if fp32 else torch.bfloat16
    tg = torch.Generator().manual_seed(7700 + seed)
    q = torch.randn(B, Hq, D, generator=tg).to(dt)
    k = torch.randn(B, Hkv, D, generator=tg).to(dt)
    v = torch.randn(B, Hkv, D, generator=tg).to(dt)
    kr0 = torch.randn(B, Hkv, W, D, generator=tg).to(dt)
    vr0 = torch.randn(B, Hkv, W, D, generator=tg).to(dt)
    pos = torch.from_numpy(g.integers(-2, 1 << 19, size=B)).to(torch.int64)
    kr, vr = kr0.cuda(), vr0.cuda()
    q_out = torch.full((B, Hq, D), 7.0, dtype=dt, device="cuda")
    swa.swa_rope_append(q.cuda(), k.cuda(), v.cuda(), kr, vr, pos.cuda(), rot, theta, q_out=q_out)
    torch.cuda.synchronize()
    pos_ok = pos.clamp(min=0)
    q_ref = oracle.rope(q.unsqueeze(1), pos_ok, rot, theta)[:, 0]
    k_ref = oracle.rope(k.unsqueeze(1), pos_ok, rot, theta)[:, 0]
    kr_h, vr_h, qo_h = kr.cpu(), vr.cpu(), q_out.cpu()
    for b in range(B):
        p = int(pos[b])
        if p < 0:   # a negative position writes nothing
            assert torch.equal(kr_h[b], kr0[b]) and torch.equal(vr_h[b], vr0[b])
            assert torch.all(qo_h[b] == 7.0)
            continue
        s = p % W
        _rope_close(qo_h[b].double().numpy(), q_ref[b], fp32)
        _rope_close(kr_h[b, :, s].double().numpy(), k_ref[b], fp32)
        assert torch.equal(vr_h[b, :, s], v[b])
        keep = [t for t in range(W) if t != s]
        assert torch.equal(kr_h[b][:, keep], kr0[b][:, keep])
        assert torch.equal(vr_h[b][:, keep], vr0[b][:, keep])
    assert swa.device_error() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_ring_append_shape(cuda_ok, seed):
    g = np.random.default_rng(7800 + seed)
    D = int(g.choice((64, 128)))
    B, Hkv, W = int(g.integers(1, 60)), int(g.integers(1, 9)), int(g.choice((1, 33, 128, 200)))
    dt = torch.float32 if g.random() < 0.5 else torch.bfloat16
    tg = torch.Generator().manual_seed(7800 + seed)
    k = torch.randn(B, Hkv, D, generator=tg).to(dt)
    v = torch.randn(B, Hkv, D, generator=tg).to(dt)
    kr0 = torch.randn(B, Hkv, W, D, generator=tg).to(dt)
    vr0 = torch.randn(B, Hkv, W, D, generator=tg).to(dt)
    pos = torch.from_numpy(g.integers(-2, 1 << 19, size=B)).to(torch.int64)
    kr, vr = kr0.cuda(), vr0.cuda()
    swa.swa_ring_append(k.cuda(), v.cuda(), kr, vr, pos.cuda())
    torch.cuda.synchronize()
    # expected: slot pos mod W of each sequence replaced (bit for bit), the
    # rest unchanged; a negative position writes nothing
    ek, ev = kr0.clone(), vr0.clone()
    for b in range(B):
        p = int(pos[b])
        if p >= 0:
            ek[b, :, p % W] = k[b]
            ev[b, :, p % W] = v[b]
    assert torch.equal(kr.cpu(), ek) and torch.equal(vr.cpu(), ev)
    assert swa.device_error() == 0
