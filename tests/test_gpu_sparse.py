"""High Sparse on the GPU: block scores from the global kernel, block
selection, and attention over the selected blocks, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen
from gpu_helpers import (assert_bf16_close, assert_lse_close, gather_rows,
                         oracle_block_scores_from_slices, oracle_rows_from_slices,
                         oracle_sparse_rows_from_slices)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,T,Hq,Hkv,W,D", [(1, 300, 8, 1, 300, 128), (2, 1000, 16, 2, 1000, 128),
                                            (1, 700, 8, 1, 200, 128), (1, 130, 8, 1, 130, 128),
                                            (2, 900, 16, 2, 900, 64)])
def test_block_scores_match_oracle(cuda_ok, B, T, Hq, Hkv, W, D):
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=4000 + T + W)
    q, k, v, s = (t.cuda() for t in (x.q, x.k, x.v, x.sink))
    out, lse, bm = swa.swa_sink_fwd_scores(q, k, v, s, W)
    o2, l2 = swa.swa_sink_fwd(q, k, v, s, W)
    torch.cuda.synchronize()
    if W > 129:      # same kernel with and without scores: same results
        assert torch.equal(out, o2) and torch.equal(lse, l2)
    ref = oracle.block_max(x.q, x.k, W)
    got = bm.cpu().double().numpy()
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    fin = np.isfinite(ref)
    assert np.abs(got[fin] - ref[fin]).max() <= 1e-3


@pytest.mark.parametrize("T,QB,topk", [(1000, 64, 3), (4096, 128, 8), (700, 32, 1),
                                       (3000, 4, 9), (32768, 64, 16)])
def test_topk_matches_oracle_bit_exact(cuda_ok, T, QB, topk):
    g = np.random.default_rng(T + QB + topk)
    nqg, nkb = (T + 3) // 4, (T + 127) // 128
    sc = g.normal(size=(2, 3, nqg, nkb)).astype(np.float32)
    sc[..., 3] = sc[..., 5]                         # ties
    sc[0, 0, :, 2] = -np.inf                        # a block with no valid pair
    idx = swa.swa_topk_blocks(torch.from_numpy(sc).cuda(), T, QB, topk)
    torch.cuda.synchronize()
    ref = oracle.topk_blocks(sc, T, QB, topk)
    assert np.array_equal(idx.cpu().numpy(), ref)


def _selection(B, Hkv, T, QB, topk, seed):
    g = np.random.default_rng(seed)
    sc = g.normal(size=(B, Hkv, (T + 3) // 4, (T + 127) // 128)).astype(np.float32)
    return oracle.topk_blocks(sc, T, QB, topk)


@pytest.mark.parametrize("B,T,Hq,Hkv,QB,topk,D", [(1, 600, 8, 1, 64, 2, 128), (2, 1000, 16, 2, 32, 3, 128),
                                                  (1, 1500, 8, 1, 128, 4, 128), (2, 1100, 16, 2, 64, 3, 64)])
def test_sparse_matches_oracle(cuda_ok, B, T, Hq, Hkv, QB, topk, D):
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=4100 + T)
    idx = _selection(B, Hkv, T, QB, topk, seed=T)
    q, k, v, s = (t.cuda() for t in (x.q, x.k, x.v, x.sink))
    out, lse = swa.swa_sink_sparse_fwd(q, k, v, s, torch.from_numpy(idx).cuda(), QB)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.sparse_fwd(x.q, x.k, x.v, x.sink, idx, QB)
    assert_bf16_close(out.cpu().numpy(), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)


def test_sparse_block_list_is_read_up_to_its_first_negative_entry(cuda_ok):
    # a caller-built list: entries after the first -1 are ignored, and the
    # order of the entries before it does not matter (every key is masked
    # causally on its own, and the online softmax does not depend on order)
    B, T, Hq, Hkv, QB, topk = 1, 1000, 16, 2, 64, 4
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=4150)
    idx = _selection(B, Hkv, T, QB, topk, seed=77)
    cut = idx.copy()
    cut[..., 1] = -1                       # valid entries after it are dropped
    want = cut.copy()
    want[..., 2:] = -1
    rev = idx.copy()
    for b in range(B):
        for g in range(Hkv):
            for qb in range(idx.shape[2]):
                n = int((idx[b, g, qb] >= 0).sum())
                rev[b, g, qb, :n] = idx[b, g, qb, :n][::-1]
    q, k, v, s = (t.cuda() for t in (x.q, x.k, x.v, x.sink))
    for given, ref_idx in ((cut, want), (rev, idx)):
        out, lse = swa.swa_sink_sparse_fwd(q, k, v, s, torch.from_numpy(given).cuda(), QB)
        torch.cuda.synchronize()
        o_ref, l_ref = oracle.sparse_fwd(x.q, x.k, x.v, x.sink, ref_idx, QB)
        assert_bf16_close(out.cpu().numpy(), o_ref)
        assert_lse_close(lse.cpu().numpy(), l_ref)
    assert swa.device_error() == 0


@pytest.mark.parametrize("QB,D", [(64, 128), (32, 64), (128, 128)])
def test_sparse_empty_block_lists_give_the_sink_alone(cuda_ok, QB, D):
    # a list that starts with -1 selects no key: those rows get out = 0 and
    # lse = sink (no wait runs out, and the items after them are unaffected)
    B, T, Hq, Hkv = 2, 1100, 16, 2
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=4170 + QB)
    idx = _selection(B, Hkv, T, QB, 3, seed=QB)
    idx[0, 0, 0, :] = -1                 # the first query block
    idx[0, 1, 3:6, :] = -1               # consecutive empty lists
    idx[1, :, -1, :] = -1                # the last (ragged) query block
    q, k, v, s = (t.cuda() for t in (x.q, x.k, x.v, x.sink))
    out, lse = swa.swa_sink_sparse_fwd(q, k, v, s, torch.from_numpy(idx).cuda(), QB)
    o16, l16 = swa.swa_sink_sparse_fwd(q, k, v, s, torch.from_numpy(idx).cuda(), QB,
                                       out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.sparse_fwd(x.q, x.k, x.v, x.sink, idx, QB)
    assert_bf16_close(out.cpu().numpy(), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)
    assert torch.equal(o16, out.to(torch.bfloat16)) and torch.equal(l16, lse)
    assert swa.device_error() == 0


def test_sparse_with_every_block_is_the_global_kernel(cuda_ok):
    B, T, Hq, Hkv, QB = 1, 1100, 16, 2, 64
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=4200, device="cuda")
    nkb = (T + 127) // 128
    idx = torch.arange(nkb, dtype=torch.int32, device="cuda").expand(
        B, Hkv, (T + QB - 1) // QB, nkb).contiguous()
    o_s, l_s = swa.swa_sink_sparse_fwd(x.q, x.k, x.v, x.sink, idx, QB)
    o_g, l_g = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, T)
    torch.cuda.synchronize()
    assert torch.equal(o_s, o_g) and torch.equal(l_s, l_g)


def test_scores_select_sparse_pipeline(cuda_ok):
    # global layer -> block scores -> selection -> sparse layer on the shared
    # K/V: the selection agrees with the oracle's from the same fp32 scores,
    # the sparse layer with the oracle given that selection
    B, T, Hq, Hkv, QB, topk = 1, 2048, 16, 2, 64, 4
    x = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=4300, device="cuda")
    _, _, bm = swa.swa_sink_fwd_scores(x.q, x.k, x.v, x.sink, T)
    idx = swa.swa_topk_blocks(bm, T, QB, topk)
    q2 = gen.prefill_inputs(B, T, Hq, Hkv, 128, seed=4301, device="cuda").q   # next layer's queries
    out, lse = swa.swa_sink_sparse_fwd(q2, x.k, x.v, x.sink, idx, QB)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), oracle.topk_blocks(bm.cpu().numpy(), T, QB, topk))
    o_ref, l_ref = oracle.sparse_fwd(q2.cpu(), x.k.cpu(), x.v.cpu(), x.sink.cpu(),
                                     idx.cpu().numpy(), QB)
    assert_bf16_close(out.cpu().numpy(), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)
    assert swa.device_error() == 0


def test_high_sparse_full_size_sampled(cuda_ok):
    # the High Sparse workload at full size (one sequence of T = 32768, Hq 64,
    # Hkv 8, top-16 blocks per 64-position query block, the inputs' seeds as
    # in the bench), in the same calls: scores, selection, sparse layer
    T, Hq, Hkv, D, QB, topk = 32768, 64, 8, 128, 64, 16
    x = gen.prefill_inputs(1, T, Hq, Hkv, D, seed=500, device="cuda")
    q2 = gen.prefill_inputs(1, T, Hq, Hkv, D, seed=501, device="cuda").q
    out_g, lse_g, bm = swa.swa_sink_fwd_scores(x.q, x.k, x.v, x.sink, T)
    idx = swa.swa_topk_blocks(bm, T, QB, topk)
    out, lse = swa.swa_sink_sparse_fwd(q2, x.k, x.v, x.sink, idx, QB)
    torch.cuda.synchronize()
    assert swa.device_error() == 0
    bm_h = bm.cpu().numpy()
    idx_h = idx.cpu().numpy()
    # every entry: -inf exactly where the query group has no causal key in the block
    last = 4 * np.arange(T // 4) + 3
    has_pair = (128 * np.arange(T // 128))[None, :] <= last[:, None]
    assert np.array_equal(np.isfinite(bm_h[0]), np.broadcast_to(has_pair, bm_h[0].shape))
    # the selection from these fp32 scores, bit for bit
    assert np.array_equal(idx_h, oracle.topk_blocks(bm_h, T, QB, topk))
    # sampled scores
    g = np.random.default_rng(17)
    entries = [(0, 0, 0), (0, T // 4 - 1, 0), (0, T // 4 - 1, T // 128 - 1), (0, 4095, 127)]
    for _ in range(40):
        gg = int(g.integers(0, T // 4))
        entries.append((0, gg, int(g.integers(0, (4 * gg + 3) // 128 + 1))))
    ref = oracle_block_scores_from_slices(x.q, x.k, entries)
    got = np.array([bm_h[0, :, gg, kb] for _, gg, kb in entries])
    assert np.abs(got - ref).max() <= 1e-3
    # sampled rows of the global layer that emitted the scores
    rows = [(0, h, i) for i in (0, 4095, 16383, T - 1) for h in range(0, Hq, 9)]
    o_ref, l_ref = oracle_rows_from_slices(x.q, x.k, x.v, x.sink, T, rows)
    o, l = gather_rows(out_g, lse_g, rows)
    assert_bf16_close(o, o_ref, what="global layer with scores")
    assert_lse_close(l, l_ref)
    # sampled rows of the sparse layer
    rows = [(0, 0, 0), (0, Hq - 1, T - 1), (0, 17, QB - 1), (0, 40, QB)]
    rows += [(0, int(g.integers(0, Hq)), int(g.integers(0, T))) for _ in range(60)]
    o_ref, l_ref = oracle_sparse_rows_from_slices(q2, x.k, x.v, x.sink, idx_h, QB,
                                                  [(0, h, i) for _, h, i in rows])
    o, l = gather_rows(out, lse, rows)
    assert_bf16_close(o, o_ref, what="sparse layer")
    assert_lse_close(l, l_ref)
    del x, q2, out_g, lse_g, bm, out, lse
    torch.cuda.empty_cache()
