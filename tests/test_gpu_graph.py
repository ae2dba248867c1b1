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
    outs = {}

    def calls():
        outs["dec"] = swa.swa_sink_decode(d.q, d.k_ring, d.v_ring, d.pos, d.sink, stream=st)
        outs["swa"] = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, 128, stream=st)
        outs["glb"] = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, 700, stream=st)
        outs["ver"] = swa.swa_sink_verify(vi.q, vi.k_new, vi.v_new, vi.k_ring, vi.v_ring, vi.pos,
                                          vi.sink, stream=st)

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
