"""The library's calls can be captured in a CUDA graph once each kernel has run
on the device (the first call sets its shared-memory attribute), and a replay
gives the eager result bit for bit."""
import pytest
import torch

import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen

pytestmark = pytest.mark.gpu


def test_graph_replay_equals_eager(cuda_ok):
    dev = torch.device("cuda")
    st = torch.cuda.Stream()
    d = gen.decode_inputs(64, 64, 8, 128, 128, seed=81, device=dev)
    x = gen.prefill_inputs(1, 700, 64, 8, 128, seed=82, device=dev)
    vi = gen.verify_inputs(32, 4, 64, 8, 128, 128, seed=83, device=dev)
    # the other instantiations: 16 and 4 heads per kv head, 8 drafted tokens
    d16 = gen.decode_inputs(48, 64, 4, 128, 128, seed=84, device=dev)
    x4 = gen.prefill_inputs(1, 500, 16, 4, 128, seed=85, device=dev)
    x16 = gen.prefill_inputs(1, 500, 64, 4, 128, seed=86, device=dev)
    v8 = gen.verify_inputs(24, 8, 64, 8, 128, 128, seed=87, device=dev)
    # head dimension 64: prefill, global layer, decode and verify
    x64 = gen.prefill_inputs(1, 600, 16, 2, 64, seed=88, device=dev)
    d64 = gen.decode_inputs(40, 64, 8, 64, 128, seed=89, device=dev)
    v64 = gen.verify_inputs(20, 4, 64, 8, 64, 128, seed=90, device=dev)
    outs = {}

    def calls():
        outs["dec"] = swa.swa_sink_decode(d.q, d.k_ring, d.v_ring, d.pos, d.sink, stream=st)
        outs["swa"] = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, 128, stream=st)
        outs["glb"] = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, 700, stream=st)
        outs["ver"] = swa.swa_sink_verify(vi.q, vi.k_new, vi.v_new, vi.k_ring, vi.v_ring, vi.pos,
                                          vi.sink, stream=st)
        outs["dec16"] = swa.swa_sink_decode(d16.q, d16.k_ring, d16.v_ring, d16.pos, d16.sink,
                                            stream=st)
        outs["swa4"] = swa.swa_sink_fwd(x4.q, x4.k, x4.v, x4.sink, 128, stream=st)
        outs["glb4"] = swa.swa_sink_fwd(x4.q, x4.k, x4.v, x4.sink, 500, stream=st)
        outs["swa16"] = swa.swa_sink_fwd(x16.q, x16.k, x16.v, x16.sink, 128, stream=st)
        outs["glb16"] = swa.swa_sink_fwd(x16.q, x16.k, x16.v, x16.sink, 500, stream=st)
        outs["ver8"] = swa.swa_sink_verify(v8.q, v8.k_new, v8.v_new, v8.k_ring, v8.v_ring, v8.pos,
                                           v8.sink, stream=st)
        outs["swa64"] = swa.swa_sink_fwd(x64.q, x64.k, x64.v, x64.sink, 128, stream=st)
        outs["glb64"] = swa.swa_sink_fwd(x64.q, x64.k, x64.v, x64.sink, 600, stream=st)
        outs["dec64"] = swa.swa_sink_decode(d64.q, d64.k_ring, d64.v_ring, d64.pos, d64.sink,
                                            stream=st)
        outs["ver64"] = swa.swa_sink_verify(v64.q, v64.k_new, v64.v_new, v64.k_ring, v64.v_ring,
                                            v64.pos, v64.sink, stream=st)

    with torch.cuda.stream(st):
        calls()
    torch.cuda.synchronize()
    eager = {k: (o.clone(), l.clone()) for k, (o, l) in outs.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        calls()
    for k in outs:
        outs[k][0].zero_()
        outs[k][1].zero_()
    g.replay()
    torch.cuda.synchronize()
    for k, (o, l) in outs.items():
        assert torch.equal(o, eager[k][0]), k
        assert torch.equal(l, eager[k][1]), k
    assert swa.device_error() == 0
