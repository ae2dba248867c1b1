"""The oracle-on-slices helpers that give sampled expected values at full size
(block scores and sparse-layer rows) agree with the oracle run on the whole
input, on problems small enough for the latter."""
import numpy as np
import torch

import oracle
from hybrid_sliding_window_02_b300 import inputs as gen
from gpu_helpers import oracle_block_scores_from_slices, oracle_sparse_rows_from_slices


def test_block_scores_from_slices_equal_whole_oracle():
    B, T, Hq, Hkv, D = 2, 600, 16, 2, 128
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=31)
    whole = oracle.block_max(x.q, x.k, T)
    g = np.random.default_rng(3)
    entries = [(0, 0, 0), (1, T // 4 - 1, 0), (1, T // 4 - 1, (T - 1) // 128), (0, 31, 0),
               (0, 32, 1), (0, 33, 1), (1, 63, 1), (0, 64, 1)]
    for _ in range(30):
        gg = int(g.integers(0, T // 4))
        entries.append((int(g.integers(0, B)), gg, int(g.integers(0, (4 * gg + 3) // 128 + 1))))
    got = oracle_block_scores_from_slices(x.q, x.k, entries)
    ref = np.array([whole[b, :, gg, kb] for b, gg, kb in entries])
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_sparse_rows_from_slices_equal_whole_oracle():
    B, T, Hq, Hkv, D, QB, topk = 1, 700, 16, 2, 128, 64, 3
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=32)
    sc = np.random.default_rng(4).normal(size=(B, Hkv, (T + 3) // 4, (T + 127) // 128))
    idx = oracle.topk_blocks(sc.astype(np.float32), T, QB, topk)
    o_whole, l_whole = oracle.sparse_fwd(x.q, x.k, x.v, x.sink, idx, QB)
    g = np.random.default_rng(5)
    rows = [(0, 0, 0), (0, Hq - 1, T - 1), (0, 7, 63), (0, 8, 64), (0, 3, 127), (0, 12, 128)]
    rows += [(0, int(g.integers(0, Hq)), int(g.integers(0, T))) for _ in range(30)]
    o, l = oracle_sparse_rows_from_slices(x.q, x.k, x.v, x.sink, idx, QB, rows)
    o_ref = np.array([o_whole[b, i, h] for b, h, i in rows])
    l_ref = np.array([l_whole[b, h, i] for b, h, i in rows])
    assert np.allclose(o, o_ref, rtol=0, atol=1e-12)
    assert np.allclose(l, l_ref, rtol=0, atol=1e-12)


def test_sparse_rows_from_slices_with_no_selected_key():
    # a row whose selected blocks all lie after it: out = 0, lse = sink
    B, T, Hq, Hkv, D, QB = 1, 300, 8, 1, 128, 64
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=33)
    idx = np.full((B, Hkv, (T + QB - 1) // QB, 2), -1, dtype=np.int32)
    idx[0, 0, 2] = [1, -1]                      # rows 128..191: block 1 (keys 128..255)
    o_whole, l_whole = oracle.sparse_fwd(x.q, x.k, x.v, x.sink, idx, QB)
    rows = [(0, 3, 10), (0, 5, 130)]            # query block 0 selects nothing
    o, l = oracle_sparse_rows_from_slices(x.q, x.k, x.v, x.sink, idx, QB, rows)
    assert np.all(o[0] == 0.0) and l[0] == float(x.sink[3])
    assert np.allclose(o[1], o_whole[0, 130, 5], atol=1e-12)
    assert np.allclose(l, [l_whole[0, 3, 10], l_whole[0, 5, 130]], atol=1e-12)


def test_prefill_by_slices_equal_whole_oracle():
    # the oracle on positions s0-W+1 .. s1-1 gives rows s0 .. s1-1 exactly
    from gpu_helpers import oracle_by_slices
    B, T, Hq, Hkv, D = 2, 300, 8, 2, 64
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=33)
    for W in (1, 32, 128, T):
        o_all, l_all = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
        for b, s0, s1 in ((0, 0, 100), (1, 100, 233), (1, 233, T), (0, 7, 8)):
            o, l = oracle_by_slices(x.q, x.k, x.v, x.sink, W, b, s0, s1)
            assert np.array_equal(o, o_all[b, s0:s1]) and np.array_equal(l, l_all[b, :, s0:s1])
