"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties the oracle to a fact the pages or the mathematics fix:

* brute force with an explicit T x T score matrix plus one sink column
  (numpy, fp64) on tiny inputs;
* sink -> -inf reduces to ordinary windowed softmax attention, checked against
  torch's scaled_dot_product_attention with a band mask (a library routine);
* W >= T is full causal attention ("MiMo-V2-Flash Technical Report" summary,
  前置知识 / 混合注意力机制: a global layer attends to the whole sequence),
  checked against scaled_dot_product_attention(is_causal=True);
* sink -> +inf drives the output to zero, with |o| ~ exp(-s_h);
* weights plus the sink weight sum to one per row (the sink only adds to the
  denominator: same page, 注意力sink偏置);
* W = 1 has the closed form o_i = v_i * sigmoid(x_ii - s_h);
* decode against a ring built from a history equals the prefill row at pos
  ("pwwt.cn" essay 1.1: fixed O(W) cache; ICML 2026 talk write-up, Q&A K:
  positions keep increasing while the window slides);
* keys outside the window, set to NaN, change nothing;
* the GQA grouping is contiguous (query head h reads kv head h // (Hq/Hkv));
* bf16 inputs are widened exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from hybrid_sliding_window_02_b300 import inputs as gen


def _f64(t):
    return t.detach().cpu().double().numpy()


def brute_force(q, k, v, sink, W):
    """Explicit-matrix attention: scores with -inf outside the causal band, one
    extra column holding s_h whose value row is zero."""
    q, k, v, sink = _f64(q), _f64(k), _f64(v), np.asarray(_f64(sink))
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, T, Hq, D))
    lse = np.zeros((B, Hq, T))
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    band = (j <= i) & (j > i - W)
    for b in range(B):
        for h in range(Hq):
            S = q[b, :, h, :] @ k[b, :, h // G, :].T / math.sqrt(D)
            S = np.where(band, S, -np.inf)
            S_ext = np.concatenate([S, np.full((T, 1), sink[h])], axis=1)
            V_ext = np.concatenate([v[b, :, h // G, :], np.zeros((1, D))], axis=0)
            mx = S_ext.max(axis=1, keepdims=True)
            P = np.exp(S_ext - mx)
            Z = P.sum(axis=1, keepdims=True)
            out[b, :, h, :] = (P / Z) @ V_ext
            lse[b, h, :] = (mx + np.log(Z))[:, 0]
    return out, lse


def sdpa(q, k, v, mask=None, causal=False):
    """torch SDPA in fp64 on [B,T,H,D] tensors with contiguous GQA groups."""
    q, k, v = (torch.as_tensor(_f64(x)) for x in (q, k, v))
    G = q.shape[2] // k.shape[2]
    qt = q.transpose(1, 2)
    kt = k.repeat_interleave(G, dim=2).transpose(1, 2)
    vt = v.repeat_interleave(G, dim=2).transpose(1, 2)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                         is_causal=causal)
    return o.transpose(1, 2).numpy()


@pytest.mark.parametrize("T,W", [(1, 1), (7, 1), (17, 3), (33, 8), (48, 48), (40, 45), (64, 16)])
@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (4, 2), (2, 2)])
def test_brute_force_tiny(T, W, Hq, Hkv):
    x = gen.prefill_inputs(2, T, Hq, Hkv, 16, seed=T * 7 + W, dtype=torch.float32)
    o, l = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    ob, lb = brute_force(x.q, x.k, x.v, x.sink, W)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, lb, rtol=0, atol=1e-12)


def test_brute_force_bf16_d64():
    x = gen.prefill_inputs(1, 40, 8, 1, 64, seed=3, dtype=torch.bfloat16)
    o, l = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, 9)
    ob, lb = brute_force(x.q, x.k, x.v, x.sink, 9)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("W", [1, 5, 16])
def test_sink_minus_inf_is_windowed_softmax(W):
    T = 40
    x = gen.prefill_inputs(2, T, 4, 2, 32, seed=11, dtype=torch.float32)
    sink = torch.full((4,), -math.inf)
    o, l = oracle.swa_sink_fwd(x.q, x.k, x.v, sink, W)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    band = (j <= i) & (j > i - W)
    ref = sdpa(x.q, x.k, x.v, mask=band)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    # lse is then the plain log-sum-exp of the in-window scores
    q, k = _f64(x.q), _f64(x.k)
    for h in range(4):
        S = q[0, :, h] @ k[0, :, h // 2].T / math.sqrt(32)
        S = np.where(band.numpy(), S, -np.inf)
        ref_l = np.log(np.exp(S - S.max(1, keepdims=True)).sum(1)) + S.max(1)
        np.testing.assert_allclose(l[0, h], ref_l, rtol=0, atol=1e-12)
    # a very negative finite sink agrees too
    o2, _ = oracle.swa_sink_fwd(x.q, x.k, x.v, torch.full((4,), -1e30), W)
    np.testing.assert_allclose(o2, ref, rtol=0, atol=1e-12)


def test_global_layer_is_full_causal():
    T = 48
    x = gen.prefill_inputs(2, T, 8, 2, 32, seed=5, dtype=torch.float32)
    sink = torch.full((8,), -math.inf)
    o, _ = oracle.swa_sink_fwd(x.q, x.k, x.v, sink, T)
    ref = sdpa(x.q, x.k, x.v, causal=True)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    # every W >= T gives the identical result, with the sink too
    a = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, T)
    for W in (T + 1, T + 5, 1 << 30):
        b = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # and W < T really differs from the global layer
    c = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, T - 8)
    assert not np.allclose(a[0], c[0])


def test_sink_plus_inf_limit():
    x = gen.prefill_inputs(1, 24, 4, 1, 16, seed=2, dtype=torch.float32)
    o, l = oracle.swa_sink_fwd(x.q, x.k, x.v, torch.full((4,), 1e4), 8)
    assert np.all(o == 0.0)
    assert np.all(l == 1e4)
    # |o| decays like exp(-s_h): o(s) * e^s converges as s grows
    o30, _ = oracle.swa_sink_fwd(x.q, x.k, x.v, torch.full((4,), 30.0), 8)
    o40, _ = oracle.swa_sink_fwd(x.q, x.k, x.v, torch.full((4,), 40.0), 8)
    a, b = o30 * math.exp(30.0), o40 * math.exp(40.0)
    assert np.max(np.abs(a - b)) <= 1e-8 * np.max(np.abs(b))
    assert np.max(np.abs(o40)) < 1e-14


def test_weights_plus_sink_sum_to_one():
    T, W, D = 50, 7, 32
    x = gen.prefill_inputs(2, T, 4, 2, D, seed=9, dtype=torch.float32)
    _, l = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    q, k, s = _f64(x.q), _f64(x.k), _f64(x.sink)
    for b in range(2):
        for h in range(4):
            for i in range(T):
                j0 = max(0, i - W + 1)
                sc = k[b, j0:i + 1, h // 2] @ q[b, i, h] / math.sqrt(D)
                tot = np.exp(sc - l[b, h, i]).sum() + math.exp(s[h] - l[b, h, i])
                assert abs(tot - 1.0) < 1e-12


def test_window_one_closed_form():
    T, D = 30, 16
    x = gen.prefill_inputs(1, T, 2, 1, D, seed=4, dtype=torch.float32)
    o, l = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, 1)
    q, k, v, s = _f64(x.q), _f64(x.k), _f64(x.v), _f64(x.sink)
    for h in range(2):
        for i in range(T):
            xi = q[0, i, h] @ k[0, i, 0] / math.sqrt(D)
            sig = 1.0 / (1.0 + math.exp(-(xi - s[h])))
            np.testing.assert_allclose(o[0, i, h], v[0, i, 0] * sig, rtol=0, atol=1e-13)
            lse_ref = max(xi, s[h]) + math.log1p(math.exp(-abs(xi - s[h])))
            assert abs(l[0, h, i] - lse_ref) < 1e-13


def test_gqa_grouping_is_contiguous():
    x = gen.prefill_inputs(1, 20, 6, 2, 16, seed=8, dtype=torch.float32)
    a = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, 6)
    kk = x.k.repeat_interleave(3, dim=2)
    vv = x.v.repeat_interleave(3, dim=2)
    b = oracle.swa_sink_fwd(x.q, kk, vv, x.sink, 6)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_sink_is_per_query_head():
    x = gen.prefill_inputs(1, 20, 4, 1, 16, seed=12, dtype=torch.float32)
    a, la = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, 5)
    s2 = x.sink.clone()
    s2[2] += 3.0
    b, lb = oracle.swa_sink_fwd(x.q, x.k, x.v, s2, 5)
    for h in range(4):
        same = np.array_equal(a[:, :, h], b[:, :, h]) and np.array_equal(la[:, h], lb[:, h])
        assert same == (h != 2)


def test_bf16_inputs_widen_exactly():
    x = gen.prefill_inputs(1, 24, 4, 2, 16, seed=6, dtype=torch.bfloat16)
    a = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, 5)
    b = oracle.swa_sink_fwd(x.q.float(), x.k.float(), x.v.float(), x.sink, 5)
    c = oracle.swa_sink_fwd(x.q.double(), x.k.double(), x.v.double(), x.sink, 5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[0], c[0])
    assert np.array_equal(a[1], b[1])


@pytest.mark.parametrize("W", [1, 4, 8])
def test_poisoned_keys_outside_window(W):
    T = 24
    x = gen.prefill_inputs(1, T, 2, 1, 16, seed=13, dtype=torch.float32)
    ref, lref = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    for i in (0, 3, W - 1, W, T - 1):
        if i >= T:
            continue
        k, v = x.k.clone(), x.v.clone()
        outside = [j for j in range(T) if not (i - W + 1 <= j <= i)]
        k[:, outside] = float("nan")
        v[:, outside] = float("nan")
        o, l = oracle.swa_sink_fwd_rows(x.q, k, v, x.sink, W, [[0, h, i] for h in range(2)])
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
        for h in range(2):
            assert np.array_equal(o[h], ref[0, i, h]) and l[h] == lref[0, h, i]


def test_rows_entry_matches_full():
    x = gen.prefill_inputs(2, 33, 4, 2, 16, seed=14, dtype=torch.bfloat16)
    o, l = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, 8)
    rows = [[b, h, i] for b in range(2) for h in range(4) for i in (0, 7, 8, 32)]
    orow, lrow = oracle.swa_sink_fwd_rows(x.q, x.k, x.v, x.sink, 8, rows)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(orow[n], o[b, i, h]) and lrow[n] == l[b, h, i]


@pytest.mark.parametrize("W", [1, 5, 8])
def test_decode_equals_prefill_row(W):
    B, T, Hq, Hkv, D = 3, 29, 4, 2, 16
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=21 + W, dtype=torch.bfloat16)
    o_pre, l_pre = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    for pos_list in ([0, 1, 2], [W - 1, W, W + 1], [T - 1, 13, 2 * W + 3]):
        pos = torch.tensor([min(p, T - 1) for p in pos_list], dtype=torch.int64)
        kr, vr = gen.ring_from_history(x.k, x.v, pos, W)
        qd = torch.stack([x.q[b, int(pos[b])] for b in range(B)])
        o, l = oracle.swa_sink_decode(qd, kr, vr, pos, x.sink)
        for b in range(B):
            p = int(pos[b])
            np.testing.assert_allclose(o[b], o_pre[b, p], rtol=0, atol=1e-12)
            np.testing.assert_allclose(l[b], l_pre[b, :, p], rtol=0, atol=1e-12)


def test_decode_ignores_empty_slots():
    W = 8
    x = gen.decode_inputs(4, 4, 1, 16, W, seed=1, dtype=torch.float32, pos_lo=0, pos_hi=W)
    ref = oracle.swa_sink_decode(x.q, x.k_ring, x.v_ring, x.pos, x.sink)
    k, v = x.k_ring.clone(), x.v_ring.clone()
    for b in range(4):
        for s in range(W):
            if s > int(x.pos[b]):          # slot s would hold a negative position
                k[b, :, s] = float("nan")
                v[b, :, s] = float("nan")
    got = oracle.swa_sink_decode(x.q, k, v, x.pos, x.sink)
    assert np.all(np.isfinite(got[0]))
    assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])


def test_decode_slot_mapping_wraps():
    # pos = 10, W = 4: slots 0..3 hold positions 8, 9, 10, 7 -- the ring order
    # must not matter, only which positions are present.
    B, T, Hq, Hkv, D, W = 1, 11, 2, 1, 16, 4
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=31, dtype=torch.float32)
    pos = torch.tensor([10])
    kr, vr = gen.ring_from_history(x.k, x.v, pos, W)
    for s, p in zip(range(4), (8, 9, 10, 7)):
        assert torch.equal(kr[0, :, s], x.k[0, p])
    o, l = oracle.swa_sink_decode(x.q[:, 10], kr, vr, pos, x.sink)
    ob, lb = brute_force(x.q, x.k, x.v, x.sink, W)
    np.testing.assert_allclose(o[0], ob[0, 10], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l[0], lb[0, :, 10], rtol=0, atol=1e-12)


def _verify_case(x, pos, L, W):
    """Split a history into (ring before pos, L new tokens) for each sequence."""
    B = x.q.shape[0]
    kr, vr = gen.ring_from_history(x.k, x.v, pos - 1, W)
    idx = [torch.arange(int(p), int(p) + L) for p in pos]
    qn = torch.stack([x.q[b, idx[b]] for b in range(B)])
    kn = torch.stack([x.k[b, idx[b]] for b in range(B)])
    vn = torch.stack([x.v[b, idx[b]] for b in range(B)])
    return qn, kn, vn, kr, vr


@pytest.mark.parametrize("W", [1, 3, 8])
@pytest.mark.parametrize("L", [1, 2, 4, 10])
def test_verify_equals_prefill_rows(W, L):
    # drafted tokens checked in one pass equal the prefill rows at their
    # positions: the ring carries what precedes them, the window slides on
    B, T, Hq, Hkv, D = 3, 40, 4, 2, 16
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=41 + W + L, dtype=torch.bfloat16)
    o_pre, l_pre = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    for pos_list in ([0, 1, 2], [W - 1, W, W + 1], [T - L, 13, 2 * W + 3]):
        pos = torch.tensor([max(0, min(p, T - L)) for p in pos_list], dtype=torch.int64)
        qn, kn, vn, kr, vr = _verify_case(x, pos, L, W)
        o, l = oracle.swa_sink_verify(qn, kn, vn, kr, vr, pos, x.sink)
        for b in range(B):
            p = int(pos[b])
            np.testing.assert_allclose(o[b], o_pre[b, p:p + L], rtol=0, atol=1e-12)
            np.testing.assert_allclose(l[b], l_pre[b, :, p:p + L], rtol=0, atol=1e-12)


def test_verify_one_token_is_decode_after_append():
    B, T, Hq, Hkv, D, W = 4, 30, 4, 1, 16, 8
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=51, dtype=torch.float32)
    pos = torch.tensor([0, 5, 8, 29], dtype=torch.int64)
    qn, kn, vn, kr, vr = _verify_case(x, pos, 1, W)
    o, l = oracle.swa_sink_verify(qn, kn, vn, kr, vr, pos, x.sink)
    kr2, vr2 = gen.ring_from_history(x.k, x.v, pos, W)   # token at pos appended
    od, ld = oracle.swa_sink_decode(qn[:, 0], kr2, vr2, pos, x.sink)
    np.testing.assert_allclose(o[:, 0], od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l[:, :, 0], ld, rtol=0, atol=1e-12)


def test_verify_ignores_slots_outside_every_window():
    # the slot holding pos - W is outside the window of every new token, and
    # slots of negative positions are empty: NaN there changes nothing
    B, T, Hq, Hkv, D, W, L = 3, 30, 4, 2, 16, 8, 3
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=52, dtype=torch.float32)
    pos = torch.tensor([3, 8, 20], dtype=torch.int64)
    qn, kn, vn, kr, vr = _verify_case(x, pos, L, W)
    ref = oracle.swa_sink_verify(qn, kn, vn, kr, vr, pos, x.sink)
    for b in range(B):
        p = int(pos[b])
        for s in range(W):
            ps = (p - 1) - ((p - 1 - s) % W)
            if ps < 0 or ps < p - W + 1:
                kr[b, :, s] = float("nan")
                vr[b, :, s] = float("nan")
    got = oracle.swa_sink_verify(qn, kn, vn, kr, vr, pos, x.sink)
    assert np.all(np.isfinite(got[0]))
    assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])


# ---- rotary position embedding (applied to q and k before attention) -------
def test_rope_position_zero_is_identity():
    x = torch.randn(2, 1, 3, 16, dtype=torch.float64)
    y = oracle.rope(x, torch.tensor([0, 0]), 16, 10000.0)
    np.testing.assert_array_equal(y, x.numpy())


def test_rope_two_dims_is_a_plane_rotation():
    # D = 2: (x0, x1) rotated by the angle p (theta^0 = 1)
    x = torch.tensor([[[[0.3, -1.7]]]], dtype=torch.float64).repeat(1, 5, 1, 1)
    y = oracle.rope(x, torch.tensor([7]), 2, 10000.0)
    for t in range(5):
        a = 7.0 + t
        np.testing.assert_allclose(y[0, t, 0], [0.3 * math.cos(a) + 1.7 * math.sin(a),
                                                -1.7 * math.cos(a) + 0.3 * math.sin(a)],
                                   rtol=0, atol=1e-14)


def test_rope_preserves_norms_and_passes_the_rest():
    x = torch.randn(1, 9, 2, 64, dtype=torch.float64)
    y = oracle.rope(x, torch.tensor([100000]), 48, 5e5)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x.numpy(), axis=-1),
                               rtol=1e-13)
    np.testing.assert_array_equal(y[..., 48:], x.numpy()[..., 48:])


def test_rope_scores_depend_on_relative_position_only():
    # <R(p) q, R(p') k> is a function of p - p': the property that lets the
    # window slide over absolute positions
    g = torch.Generator().manual_seed(5)
    q = torch.randn(1, 1, 1, 32, generator=g, dtype=torch.float64)
    k = torch.randn(1, 1, 1, 32, generator=g, dtype=torch.float64)
    def score(p, pk):
        return float((oracle.rope(q, torch.tensor([p]), 32, 10000.0) *
                      oracle.rope(k, torch.tensor([pk]), 32, 10000.0)).sum())
    for shift in (0, 129, 262000):
        np.testing.assert_allclose(score(shift + 40, shift + 13), score(40, 13), rtol=1e-9)


# ---- High Sparse: block scores, block selection, sparse attention ----------
def _scores_np(q, k, W):
    """Explicit scaled-logit matrix [B, Hq, T, T] with -inf outside the band."""
    q64, k64 = _f64(q), _f64(k)
    B, T, Hq, D = q64.shape
    G = Hq // k64.shape[2]
    kk = np.repeat(k64, G, axis=2)
    x = np.einsum("bihd,bjhd->bhij", q64, kk) / math.sqrt(D)
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    x[:, :, ~((j <= i) & (j > i - W))] = -np.inf
    return x


@pytest.mark.parametrize("T,W", [(10, 10), (200, 200), (300, 150), (129, 7)])
def test_block_max_is_brute_force(T, W):
    B, Hq, Hkv, D = 2, 4, 2, 16
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=91 + T, dtype=torch.float32)
    got = oracle.block_max(x.q, x.k, W)
    s = _scores_np(x.q, x.k, W)                      # [B, Hq, T, T]
    nqg, nkb = (T + 3) // 4, (T + 127) // 128
    pad = np.full((B, Hq, nqg * 4, nkb * 128), -np.inf)
    pad[:, :, :T, :T] = s
    G = Hq // Hkv
    ref = pad.reshape(B, Hkv, G, nqg, 4, nkb, 128).max(axis=(2, 4, 6))
    np.testing.assert_array_equal(np.isinf(got), np.isinf(ref))
    fin = np.isfinite(ref)
    np.testing.assert_allclose(got[fin], ref[fin], rtol=0, atol=1e-12)


def _topk_np(scores, T, QB, topk):
    B, Hkv, nqg, nkb = scores.shape
    nqb = (T + QB - 1) // QB
    out = np.full((B, Hkv, nqb, topk), -1, dtype=np.int32)
    for b in range(B):
        for g in range(Hkv):
            for qb in range(nqb):
                diag = (min(qb * QB + QB, T) - 1) // 128
                agg = scores[b, g, qb * QB // 4:(qb + 1) * QB // 4, :diag].astype(np.float64)
                agg = agg.max(axis=0) if agg.shape[0] else np.full(diag, -np.inf)
                order = np.lexsort((np.arange(diag), -agg))   # score desc, index asc
                chosen = sorted([diag] + [int(c) for c in order[:topk - 1]])
                out[b, g, qb, :len(chosen)] = chosen
    return out


@pytest.mark.parametrize("T,QB,topk", [(1000, 64, 3), (2048, 128, 5), (700, 32, 1), (300, 16, 9)])
def test_topk_blocks_matches_ranking(T, QB, topk):
    g = np.random.default_rng(T + QB + topk)
    nqg, nkb = (T + 3) // 4, (T + 127) // 128
    scores = g.normal(size=(2, 3, nqg, nkb)).astype(np.float32)
    scores[..., 1] = scores[..., 2]                  # a tie: the smaller index wins
    got = oracle.topk_blocks(scores, T, QB, topk)
    np.testing.assert_array_equal(got, _topk_np(scores, T, QB, topk))
    for b, gg, qb in np.ndindex(*got.shape[:3]):
        sel = got[b, gg, qb]
        live = sel[sel >= 0]
        diag = (min(qb * QB + QB, T) - 1) // 128
        assert diag in live and np.all(np.diff(live) > 0)
        assert len(live) == min(topk, diag + 1)


def test_sparse_with_every_block_is_the_global_layer():
    B, T, Hq, Hkv, D, QB = 2, 300, 4, 2, 16, 32
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=95, dtype=torch.bfloat16)
    nkb = (T + 127) // 128
    idx = np.tile(np.arange(nkb, dtype=np.int32), (B, Hkv, (T + QB - 1) // QB, 1))
    o, l = oracle.sparse_fwd(x.q, x.k, x.v, x.sink, idx, QB)
    og, lg = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, T)
    np.testing.assert_allclose(o, og, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, lg, rtol=0, atol=1e-12)


def test_sparse_is_brute_force_with_a_block_mask():
    B, T, Hq, Hkv, D, QB, topk = 1, 400, 4, 2, 16, 16, 2
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=96, dtype=torch.float32)
    g = np.random.default_rng(7)
    nqb, nkb = (T + QB - 1) // QB, (T + 127) // 128
    idx = np.full((B, Hkv, nqb, topk), -1, dtype=np.int32)
    for gg in range(Hkv):
        for qb in range(nqb):
            diag = (min(qb * QB + QB, T) - 1) // 128
            other = [int(c) for c in g.permutation(diag)[:topk - 1]]
            sel = sorted(set([diag] + other))
            idx[0, gg, qb, :len(sel)] = sel
    o, l = oracle.sparse_fwd(x.q, x.k, x.v, x.sink, idx, QB)
    s = _scores_np(x.q, x.k, T)                      # causal, [B, Hq, T, T]
    G = Hq // Hkv
    allowed = np.zeros((Hkv, T, T), dtype=bool)
    for gg in range(Hkv):
        for i in range(T):
            for kb in idx[0, gg, i // QB]:
                if kb >= 0:
                    allowed[gg, i, kb * 128:kb * 128 + 128] = True
    s[0][~np.repeat(allowed, G, axis=0)] = -np.inf
    sk = _f64(x.sink)[None, :, None, None]
    m = np.maximum(s.max(axis=-1, keepdims=True), sk)
    e = np.exp(s - m)
    lsum = e.sum(axis=-1, keepdims=True) + np.exp(sk - m)
    vv = np.repeat(_f64(x.v), G, axis=2)
    ref = np.einsum("bhij,bjhd->bihd", e / lsum, vv)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, (m + np.log(lsum))[..., 0], rtol=0, atol=1e-12)


def test_sparse_ignores_keys_outside_the_selection():
    B, T, Hq, Hkv, D, QB = 1, 384, 2, 1, 16, 128
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=97, dtype=torch.float32)
    idx = np.array([[[[0, -1], [1, -1], [0, 2]]]], dtype=np.int32)   # block 1 unused by qb 2
    ref = oracle.sparse_fwd(x.q, x.k, x.v, x.sink, idx, QB)
    k, v = x.k.clone(), x.v.clone()
    k[:, 128:256] = float("nan")
    v[:, 128:256] = float("nan")
    got = oracle.sparse_fwd(x.q, k, v, x.sink, idx, QB)
    np.testing.assert_array_equal(got[0][:, 256:], ref[0][:, 256:])
    np.testing.assert_array_equal(got[0][:, :128], ref[0][:, :128])
