"""swa_sink_fwd_host (prefill from and to host memory, pipelined in chunks)
against the device-buffer call and the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen
from gpu_helpers import assert_bf16_close, assert_lse_close

pytestmark = pytest.mark.gpu


def _device_call(x, W, out_dtype=torch.float32):
    out, lse = swa.swa_sink_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.sink.cuda(), W,
                                out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("B,T,Hq,Hkv,D,W", [
    (3, 300, 16, 2, 128, 128),    # sliding window: one chunk per sequence
    (1, 5000, 16, 2, 128, 128),   # 9 position chunks of 560, the last one ragged (520)
    (3, 1030, 16, 2, 128, 33),    # 2 position chunks per sequence, narrow window
    (2, 1000, 8, 1, 128, 1000),   # global layer: chunks of one sequence (Hkv = 1)
    (2, 600, 16, 2, 128, 600),    # global layer: one sequence x half the kv heads
    (1, 77, 8, 1, 128, 128),
    (2, 8192, 64, 8, 128, 128),   # the bench's shapes, two sequences: 8 chunks each
    (4, 8192, 64, 8, 128, 128),   # the bench's end-to-end workload: 4 chunks of 2048 each
    (2, 77, 3, 1, 64, 33),        # general kernel, lse slabs not 16-byte aligned: one chunk
    (2, 300, 2, 1, 128, 128),     # 2 heads per kv head, W 128: the online-softmax kernel
    (1, 5000, 16, 4, 128, 128),   # 4 heads per kv head: position chunks of whole 32-position tiles
    (2, 1500, 64, 4, 128, 128),   # 16 heads per kv head (two groups of 8)
    (2, 2600, 64, 8, 64, 128),    # head dimension 64
    (2, 900, 32, 4, 64, 900),     # head dimension 64, global layer: half the kv heads per chunk
    (2, 700, 16, 4, 128, 700),    # global layer with 4 heads per kv head
])
def test_host_call_equals_device_call(cuda_ok, pinned, B, T, Hq, Hkv, D, W):
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=B + T)
    q, k, v = (t.pin_memory() if pinned else t.clone() for t in (x.q, x.k, x.v))
    out_h, lse_h, _ = swa.swa_sink_fwd_host(q, k, v, x.sink.cuda(), W)
    torch.cuda.synchronize()
    out_d, lse_d = _device_call(x, W)
    assert torch.equal(out_h, out_d)
    assert torch.equal(lse_h, lse_d)


def test_host_call_matches_oracle_and_reuses_work(cuda_ok):
    x = gen.prefill_inputs(2, 400, 16, 2, 128, seed=3)
    q, k, v = (t.pin_memory() for t in (x.q, x.k, x.v))
    sink = x.sink.cuda()
    out_h, lse_h, work = swa.swa_sink_fwd_host(q, k, v, sink, 128)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.swa_sink_fwd(x.q, x.k, x.v, x.sink, 128)
    assert_bf16_close(out_h.double().numpy(), o_ref)
    assert_lse_close(lse_h.double().numpy(), l_ref)
    # a second call through the same device buffers, with other inputs
    y = gen.prefill_inputs(2, 400, 16, 2, 128, seed=4)
    q2, k2, v2 = (t.pin_memory() for t in (y.q, y.k, y.v))
    out2, lse2, _ = swa.swa_sink_fwd_host(q2, k2, v2, y.sink.cuda(), 128, work=work)
    torch.cuda.synchronize()
    o2, l2 = _device_call(y, 128)
    assert torch.equal(out2, o2) and torch.equal(lse2, l2)


@pytest.mark.parametrize("B,T", [(3, 256), (2, 2100)])
def test_host_call_without_lse_and_bf16_output(cuda_ok, B, T):
    x = gen.prefill_inputs(B, T, 16, 2, 128, seed=5)
    q, k, v = (t.pin_memory() for t in (x.q, x.k, x.v))
    out_h, lse_h, _ = swa.swa_sink_fwd_host(q, k, v, x.sink.cuda(), 128, with_lse=False,
                                            out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert lse_h is None and out_h.dtype == torch.bfloat16
    out_d, _ = _device_call(x, 128, out_dtype=torch.bfloat16)
    assert torch.equal(out_h, out_d)


def test_host_call_orders_with_the_stream(cuda_ok):
    # work enqueued on the same stream after the call sees the copies completed
    x = gen.prefill_inputs(2, 300, 16, 2, 128, seed=6)
    q, k, v = (t.pin_memory() for t in (x.q, x.k, x.v))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out_h, lse_h, work = swa.swa_sink_fwd_host(q, k, v, x.sink.cuda(), 128, stream=s)
        flag = torch.ones(1, device="cuda")
        flag_h = flag.to("cpu", non_blocking=True)
    s.synchronize()
    out_d, lse_d = _device_call(x, 128)
    assert flag_h.item() == 1.0
    assert torch.equal(out_h, out_d) and torch.equal(lse_h, lse_d)
    assert swa.device_error() == 0
