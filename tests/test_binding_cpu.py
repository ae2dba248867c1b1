"""Host-side checks of the Python binding, without a GPU: a caller-supplied
output buffer of the wrong shape, dtype or layout is refused before the
library is called (a kernel writes its outputs in full, so a short buffer
would be written past its end).

The device checks are relaxed to accept CPU tensors and the library call is
replaced by a recorder, so only the binding's own logic runs."""
import pytest
import torch

import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen


@pytest.fixture
def calls(monkeypatch):
    made = []

    def cuda_contig(name, t, device=None):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if device is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, expected {device}")

    monkeypatch.setattr(swa, "_cuda_contig", cuda_contig)
    monkeypatch.setattr(swa, "_call", lambda fn, dev, *args: made.append(fn))
    monkeypatch.setattr(swa, "_stream_handle", lambda stream, dev: None)
    return made


def _prefill():
    return gen.prefill_inputs(2, 40, 8, 1, 64, seed=1)


def test_prefill_outputs(calls):
    x = _prefill()
    f32, bf16 = torch.float32, torch.bfloat16
    swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, 16)
    swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, 16, out=torch.empty(2, 40, 8, 64, dtype=bf16))
    assert calls == ["swa_sink_fwd_ex"] * 2
    bad = [
        dict(out=torch.empty(2, 40, 8, 32)),                     # too short
        dict(out=torch.empty(2, 40, 8, 64, dtype=torch.float16)),
        dict(out=torch.empty(2, 40, 64, 8).transpose(2, 3)),     # not contiguous
        dict(lse=torch.empty(2, 40, 8)),                         # [B, T, Hq] instead of [B, Hq, T]
        dict(lse=torch.empty(2, 8, 40, dtype=bf16)),
        dict(lse=torch.empty(2, 8, 39)),
    ]
    for kw in bad:
        with pytest.raises(ValueError):
            swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, 16, **kw)
    assert len(calls) == 2
    assert f32 is torch.float32


def test_decode_outputs(calls):
    d = gen.decode_inputs(3, 8, 2, 64, 16, seed=2)
    swa.swa_sink_decode(d.q, d.k_ring, d.v_ring, d.pos, d.sink)
    assert calls == ["swa_sink_decode"]
    for kw in (dict(out=torch.empty(3, 8, 32)), dict(out=torch.empty(3, 8, 64, dtype=torch.bfloat16)),
               dict(lse=torch.empty(3, 4)), dict(lse=torch.empty(3, 8, dtype=torch.float64))):
        with pytest.raises(ValueError):
            swa.swa_sink_decode(d.q, d.k_ring, d.v_ring, d.pos, d.sink, **kw)
    assert len(calls) == 1


def test_verify_outputs(calls):
    v = gen.verify_inputs(2, 3, 8, 2, 64, 16, seed=3)
    args = (v.q, v.k_new, v.v_new, v.k_ring, v.v_ring, v.pos, v.sink)
    swa.swa_sink_verify(*args)
    assert calls == ["swa_sink_verify"]
    for kw in (dict(out=torch.empty(2, 3, 8, 63)), dict(out=torch.empty(2, 8, 3, 64)),
               dict(lse=torch.empty(2, 3, 8)), dict(lse=torch.empty(2, 8, 3, dtype=torch.bfloat16))):
        with pytest.raises(ValueError):
            swa.swa_sink_verify(*args, **kw)
    assert len(calls) == 1


def test_host_prefill_outputs(calls):
    x = _prefill()
    sink = x.sink
    swa.swa_sink_fwd_host(x.q, x.k, x.v, sink, 16)
    assert calls == ["swa_sink_fwd_host"]
    for kw in (dict(out_h=torch.empty(2, 40, 8, 60)),
               dict(out_h=torch.empty(2, 40, 8, 64, dtype=torch.float64)),
               dict(lse_h=torch.empty(2, 40, 8)),
               dict(lse_h=torch.empty(2, 8, 40, dtype=torch.bfloat16))):
        with pytest.raises(ValueError):
            swa.swa_sink_fwd_host(x.q, x.k, x.v, sink, 16, **kw)
    # a staging lse of the wrong shape
    work = (torch.empty_like(x.q), torch.empty_like(x.k), torch.empty_like(x.v),
            torch.empty(2, 40, 8, 64), torch.empty(2, 40, 8))
    with pytest.raises(ValueError):
        swa.swa_sink_fwd_host(x.q, x.k, x.v, sink, 16, work=work)
    assert len(calls) == 1


def test_rope_append_output(calls):
    d = gen.decode_inputs(2, 8, 2, 64, 16, seed=4)
    k_new = d.k_ring[:, :, 0].contiguous()
    swa.swa_rope_append(d.q, k_new, k_new.clone(), d.k_ring, d.v_ring, d.pos, 64, 1e4)
    assert calls == ["swa_rope_append"]
    with pytest.raises(ValueError):
        swa.swa_rope_append(d.q, k_new, k_new.clone(), d.k_ring, d.v_ring, d.pos, 64, 1e4,
                            q_out=torch.empty(2, 4, 64, dtype=d.q.dtype))
    assert len(calls) == 1
