"""Stream order across back-to-back calls of the tensor-core decode and verify
kernels, which are launched as programmatic dependents: a call may start its
set-up while the previous kernel on the stream finishes, but must read and
write nothing before that kernel has completed.  Each case below chains
calls through one buffer without synchronising in between and compares with
the same calls run one at a time."""
import pytest
import torch

import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen

pytestmark = pytest.mark.gpu

B, Hq, Hkv, D, W = 64, 64, 8, 128, 128   # 512 groups: several per CTA


def _dec(x, sink, out=None, lse=None, stream=None):
    return swa.swa_sink_decode(x.q, x.k_ring, x.v_ring, x.pos, sink, out, lse, stream=stream)


def _ver(x, sink, out=None, lse=None, stream=None):
    return swa.swa_sink_verify(x.q, x.k_new, x.v_new, x.k_ring, x.v_ring, x.pos, sink, out, lse,
                               stream=stream)


def test_read_after_write_through_the_sink(cuda_ok):
    # each call's sink is a row of the lse the call before it wrote
    dev = torch.device("cuda")
    xa = gen.decode_inputs(B, Hq, Hkv, D, W, seed=91, device=dev)
    xb = gen.decode_inputs(B, Hq, Hkv, D, W, seed=92, device=dev)
    vi = gen.verify_inputs(B, 4, Hq, Hkv, D, W, seed=93, device=dev)
    # one at a time
    _, l1 = _dec(xa, xa.sink)
    torch.cuda.synchronize()
    o2_ref, l2_ref = _dec(xb, l1[5].clone())
    torch.cuda.synchronize()
    o3_ref, l3_ref = _ver(vi, l2_ref[7].clone())
    torch.cuda.synchronize()
    o4_ref, l4_ref = _dec(xa, l3_ref[3, :, 1].contiguous())
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    for _ in range(10):
        with torch.cuda.stream(st):
            _, m1 = _dec(xa, xa.sink, stream=st)
            o2, m2 = _dec(xb, m1[5], stream=st)
            o3, m3 = _ver(vi, m2[7], stream=st)
            s4 = torch.empty(Hq, device=dev)
            s4.copy_(m3[3, :, 1])
            o4, m4 = _dec(xa, s4, stream=st)
        st.synchronize()
        assert torch.equal(o2, o2_ref) and torch.equal(m2, l2_ref)
        assert torch.equal(o3, o3_ref) and torch.equal(m3, l3_ref)
        assert torch.equal(o4, o4_ref) and torch.equal(m4, l4_ref)
    assert swa.device_error() == 0


def test_write_after_read_of_the_sink(cuda_ok):
    # a call writes its lse over the sink the call before it reads
    dev = torch.device("cuda")
    xa = gen.decode_inputs(B, Hq, Hkv, D, W, seed=94, device=dev)
    xb = gen.decode_inputs(B, Hq, Hkv, D, W, seed=95, device=dev)
    o1_ref, l1_ref = _dec(xa, xa.sink)
    o2_ref, l2_ref = _dec(xb, xb.sink)
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    for _ in range(10):
        with torch.cuda.stream(st):
            buf = torch.empty(B, Hq, device=dev)
            buf[0].copy_(xa.sink)
            o1, l1 = _dec(xa, buf[0], stream=st)
            o2, _ = _dec(xb, xb.sink, lse=buf, stream=st)
        st.synchronize()
        assert torch.equal(o1, o1_ref) and torch.equal(l1, l1_ref)
        assert torch.equal(o2, o2_ref) and torch.equal(buf, l2_ref)
    assert swa.device_error() == 0


def test_write_after_write_into_one_output(cuda_ok):
    # calls on alternating inputs into the same buffers: the last call wins
    dev = torch.device("cuda")
    xs = [gen.decode_inputs(B, Hq, Hkv, D, W, seed=96 + i, device=dev) for i in range(2)]
    vs = [gen.verify_inputs(B, 3, Hq, Hkv, D, W, seed=98 + i, device=dev) for i in range(2)]
    od_ref, ld_ref = _dec(xs[1], xs[1].sink)
    ov_ref, lv_ref = _ver(vs[1], vs[1].sink)
    torch.cuda.synchronize()
    od, ld = torch.empty_like(od_ref), torch.empty_like(ld_ref)
    ov, lv = torch.empty_like(ov_ref), torch.empty_like(lv_ref)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for _ in range(20):
            for i in range(2):
                _dec(xs[i], xs[i].sink, od, ld, stream=st)
                _ver(vs[i], vs[i].sink, ov, lv, stream=st)
    st.synchronize()
    assert torch.equal(od, od_ref) and torch.equal(ld, ld_ref)
    assert torch.equal(ov, ov_ref) and torch.equal(lv, lv_ref)
    assert swa.device_error() == 0
