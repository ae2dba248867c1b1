"""Parity at the full sizes of the bench's other-shape lines: the tensor-core
kernels with 4 and 16 query heads per kv head, at head dimension 64, and with
8 drafted tokens, every element of out and lse against the fp64 oracle (the
D = 64 global layer on sampled rows), with the inputs the bench draws (same
generators and seeds)."""
import pytest
import torch

import oracle
import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen
from gpu_helpers import (assert_bf16_close, assert_lse_close, gather_rows, oracle_by_slices,
                         oracle_rows_from_slices, sample_rows)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (64, 4, 128), (64, 8, 64)])
def test_prefill_other_group_sizes_full_size(cuda_ok, Hq, Hkv, D):
    B, T, W = 4, 8192, 128
    assert swa.fwd_path(B, T, Hq, Hkv, D, W) == "tc_swa"
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7, device="cuda")
    out, lse = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    torch.cuda.synchronize()
    for b in range(B):
        o_ref, l_ref = oracle_by_slices(x.q, x.k, x.v, x.sink, W, b, 0, T)
        assert_bf16_close(out[b].cpu().numpy(), o_ref, what=f"sequence {b}")
        assert_lse_close(lse[b].cpu().numpy(), l_ref)
    del x, out, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (64, 4, 128), (64, 8, 64)])
def test_decode_other_group_sizes_full_size(cuda_ok, Hq, Hkv, D):
    B, W = 256, 128
    assert swa.decode_path(B, Hq, Hkv, D, W) == "tc_decode"
    d = gen.decode_inputs(B, Hq, Hkv, D, W, seed=100, device="cuda")
    out, lse = swa.swa_sink_decode(d.q, d.k_ring, d.v_ring, d.pos, d.sink)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.swa_sink_decode(*(t.cpu() for t in (d.q, d.k_ring, d.v_ring, d.pos,
                                                              d.sink)))
    assert_bf16_close(out.cpu().numpy(), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)


def test_verify_eight_drafts_full_size(cuda_ok):
    B, L, Hq, Hkv, D, W = 256, 8, 64, 8, 128, 128
    assert swa.verify_path(B, L, Hq, Hkv, D, W) == "tc_verify"
    v = gen.verify_inputs(B, L, Hq, Hkv, D, W, seed=300, device="cuda")
    out, lse = swa.swa_sink_verify(v.q, v.k_new, v.v_new, v.k_ring, v.v_ring, v.pos, v.sink)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.swa_sink_verify(*(t.cpu() for t in (v.q, v.k_new, v.v_new, v.k_ring,
                                                              v.v_ring, v.pos, v.sink)))
    assert_bf16_close(out.cpu().numpy(), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)
    assert swa.device_error() == 0


def test_global_layer_head_dim_64_full_size_sampled(cuda_ok):
    # the bench's global_d64 line: B1 T16384 Hq64 Hkv8 D64, W = T (2.2e12 FLOP,
    # about two minutes of oracle in full): the 10 edge positions plus 54 drawn
    # over the whole causal range, every head
    B, T, Hq, Hkv, D = 1, 16384, 64, 8, 64
    assert swa.fwd_path(B, T, Hq, Hkv, D, T) == "tc_global"
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7, device="cuda")
    out, lse = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, T)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    rows = sample_rows(B, T, Hq, 64, seed=64)
    o_ref, l_ref = oracle_rows_from_slices(x.q, x.k, x.v, x.sink, T, rows)
    o, l = gather_rows(out, lse, rows)
    assert_bf16_close(o, o_ref)
    assert_lse_close(l, l_ref)
    assert swa.device_error() == 0
