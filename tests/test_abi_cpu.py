"""The C-ABI library without a GPU: it loads, exports what the header declares,
and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import build as swabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swasink.h")


@pytest.fixture(scope="module")
def L():
    swabuild.build()
    return swa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("swa_sink_fwd", "swa_sink_decode", "swa_ring_append", "swa_sink_verify",
                 "swa_status_str"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    assert swa.status_str(swa.SWA_OK) == "ok"
    assert swa.status_str(swa.SWA_EINVAL) == "invalid argument"
    assert swa.status_str(swa.SWA_EUNSUPPORTED) == "unsupported configuration"
    assert swa.status_str(swa.SWA_ECUDA) == "CUDA error"
    assert swa.version() >= 100


def test_path_selection(L):
    assert swa.fwd_path(4, 8192, 64, 8, 128, 128) == "tc_swa"
    assert swa.fwd_path(1, 262144, 64, 8, 128, 128) == "tc_swa"
    assert swa.fwd_path(1, 512, 64, 8, 128, 129) == "tc_swa"
    assert swa.fwd_path(1, 512, 64, 8, 128, 130) == "tc_global"
    assert swa.fwd_path(1, 32768, 64, 8, 128, 32768) == "tc_global"
    assert swa.fwd_path(1, 512, 4, 1, 64, 128, swa.SWA_F32) == "simt"
    assert swa.fwd_path(1, 512, 64, 8, 128, 128, swa.SWA_F32) == "simt"
    assert swa.fwd_path(1, 512, 64, 64, 128, 128) == "tc_global"   # 1 head per kv head: any window
    assert swa.fwd_path(1, 512, 16, 4, 128, 128) == "tc_swa"       # 4 heads per kv head
    assert swa.fwd_path(1, 512, 16, 4, 128, 130) == "tc_global"    # ... and on the global kernel
    assert swa.fwd_path(1, 512, 8, 4, 128, 512) == "tc_global"      # 2 heads per kv head
    assert swa.fwd_path(1, 512, 9, 3, 128, 512) == "simt"           # 3
    assert swa.fwd_path(1, 512, 64, 4, 128, 128) == "tc_swa"       # 16: two groups of 8
    assert swa.fwd_path(1, 512, 64, 4, 128, 512) == "tc_global"
    assert swa.fwd_path(1, 512, 48, 2, 128, 128) == "tc_swa"       # 24
    assert swa.fwd_path(1, 512, 32, 16, 128, 128) == "tc_global"   # 2 heads per kv head, W 128
    assert swa.fwd_path(1, 512, 12, 1, 128, 128) == "simt"         # 12: not a multiple of 8
    assert swa.fwd_path(1, 512, 64, 8, 64, 128) == "tc_swa"        # head dimension 64
    assert swa.fwd_path(1, 512, 16, 4, 64, 128) == "tc_swa"
    assert swa.fwd_path(1, 512, 64, 8, 64, 512) == "tc_global"     # D 64 on the global kernel
    assert swa.fwd_path(1, 512, 64, 7, 128, 128) == "invalid"
    assert swa.fwd_path(1, 512, 64, 8, 96, 128) == "invalid"
    assert swa.fwd_path(0, 512, 64, 8, 128, 128) == "invalid"


def test_decode_path_selection(L):
    assert swa.decode_path(256, 64, 8, 128, 128) == "tc_decode"
    assert swa.decode_path(256, 64, 8, 128, 128, swa.SWA_F32) == "simt_decode"
    assert swa.decode_path(256, 64, 8, 64, 128) == "tc_decode"       # head dimension 64
    assert swa.decode_path(256, 64, 8, 64, 64) == "simt_decode"      # a 64-slot ring
    assert swa.decode_path(256, 32, 8, 128, 128) == "tc_decode"      # 4 heads per kv head
    assert swa.decode_path(256, 64, 4, 128, 128) == "tc_decode"      # 16
    assert swa.decode_path(256, 8, 8, 128, 128) == "tc_decode"       # 1
    assert swa.decode_path(256, 64, 2, 128, 128) == "tc_decode"      # 32: four groups of 8
    assert swa.decode_path(256, 96, 4, 128, 128) == "tc_decode"      # 24: three groups of 8
    assert swa.decode_path(256, 48, 4, 128, 128) == "simt_decode"    # 12: not a multiple of 8
    assert swa.decode_path(256, 24, 8, 128, 128) == "simt_decode"    # 3
    assert swa.decode_path(256, 64, 8, 128, 320) == "simt_decode"
    assert swa.decode_path(256, 64, 8, 128, 321) == "invalid"
    assert swa.decode_path(256, 64, 7, 128, 128) == "invalid"


A = 1 << 20  # a fake, 16-byte aligned address: never dereferenced by these calls


def _fwd(L, q=A, k=A, v=A, sink=A, out=A, lse=A, B=1, T=16, Hq=8, Hkv=8, D=128, W=4, dt=1):
    return L.swa_sink_fwd(q, k, v, sink, out, lse, B, T, Hq, Hkv, D, W, dt, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1), (dict(k=None), -1), (dict(v=None), -1), (dict(sink=None), -1),
    (dict(out=None), -1), (dict(B=0), -1), (dict(T=0), -1), (dict(Hq=0), -1),
    (dict(Hkv=0), -1), (dict(Hq=8, Hkv=3), -1), (dict(W=0), -1), (dict(W=-5), -1),
    (dict(dt=7), -1), (dict(q=A + 8), -1), (dict(out=A + 4), -1), (dict(lse=A + 2), -1),
    (dict(D=96), -2), (dict(D=256), -2),
])
def test_fwd_rejects_before_launch(L, kw, status):
    assert _fwd(L, **kw) == status


def _dec(L, q=A, kr=A, vr=A, pos=A, sink=A, out=A, lse=A, B=2, Hq=8, Hkv=1, D=128, W=128, dt=1):
    return L.swa_sink_decode(q, kr, vr, pos, sink, out, lse, B, Hq, Hkv, D, W, dt, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1), (dict(kr=None), -1), (dict(vr=None), -1), (dict(pos=None), -1),
    (dict(sink=None), -1), (dict(out=None), -1), (dict(B=0), -1), (dict(Hq=6, Hkv=4), -1),
    (dict(W=0), -1), (dict(pos=A + 4), -1), (dict(kr=A + 8), -1), (dict(D=32), -2),
    (dict(W=321), -2), (dict(W=161, dt=0), -2),
])
def test_decode_rejects_before_launch(L, kw, status):
    assert _dec(L, **kw) == status


@pytest.mark.parametrize("args,status", [
    ((None, A, A, A, A, 1, 1, 128, 8, 1), -1),
    ((A, A, A, A, None, 1, 1, 128, 8, 1), -1),
    ((A, A, A, A, A, 0, 1, 128, 8, 1), -1),
    ((A, A, A, A, A, 1, 1, 128, 0, 1), -1),
    ((A, A, A + 4, A, A, 1, 1, 128, 8, 1), -1),
    ((A, A, A, A, A, 1, 1, 48, 8, 1), -2),
])
def test_ring_append_rejects_before_launch(L, args, status):
    assert L.swa_ring_append(*args, None) == status


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib
    mod = importlib.import_module("hybrid_sliding_window_02_b300")
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        mod.lib()


def _ver(L_, q=A, kn=A, vn=A, kr=A, vr=A, pos=A, sink=A, out=A, lse=A, B=2, L=4, Hq=8, Hkv=1,
         D=128, W=128, dt=1):
    return L_.swa_sink_verify(q, kn, vn, kr, vr, pos, sink, out, lse, B, L, Hq, Hkv, D, W, dt,
                              None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1), (dict(kn=None), -1), (dict(vn=None), -1), (dict(kr=None), -1),
    (dict(vr=None), -1), (dict(pos=None), -1), (dict(sink=None), -1), (dict(out=None), -1),
    (dict(B=0), -1), (dict(L=0), -1), (dict(Hq=6, Hkv=4), -1), (dict(W=0), -1),
    (dict(kn=A + 8), -1), (dict(pos=A + 4), -1), (dict(dt=3), -1), (dict(D=32), -2),
    (dict(L=65), -2), (dict(W=321), -2),
])
def test_verify_rejects_before_launch(L, kw, status):
    assert _ver(L, **kw) == status


def test_verify_path_selection(L):
    assert swa.verify_path(2, 4, 8, 1, 128, 128) == "tc_verify"
    assert swa.verify_path(2, 1, 64, 8, 128, 128) == "tc_verify"
    assert swa.verify_path(2, 5, 64, 8, 128, 128) == "tc_verify"
    assert swa.verify_path(2, 8, 64, 8, 128, 128) == "tc_verify"
    assert swa.verify_path(2, 9, 64, 8, 128, 128) == "simt_verify"
    assert swa.verify_path(2, 4, 64, 8, 128, 128, swa.SWA_F32) == "simt_verify"
    assert swa.verify_path(2, 4, 8, 1, 64, 128) == "tc_verify"     # head dimension 64
    assert swa.verify_path(2, 4, 8, 1, 64, 32) == "simt_verify"
    assert swa.verify_path(2, 65, 8, 1, 128, 128) == "invalid"
    assert swa.verify_path(2, 4, 64, 4, 128, 128) == "tc_verify"    # 16 heads per kv head
    assert swa.verify_path(2, 8, 96, 4, 64, 128) == "tc_verify"     # 24
    assert swa.verify_path(2, 4, 32, 8, 128, 128) == "tc_verify"    # 4
    assert swa.verify_path(2, 8, 16, 8, 64, 128) == "tc_verify"     # 2
    assert swa.verify_path(2, 8, 8, 8, 128, 128) == "tc_verify"     # 1
    assert swa.verify_path(2, 4, 24, 8, 128, 128) == "simt_verify"  # 3


@pytest.mark.parametrize("args,status", [
    ((None, A, 1, 4, 2, 128, 128, 1e4, 1), -1),
    ((A, None, 1, 4, 2, 128, 128, 1e4, 1), -1),
    ((A, A, 0, 4, 2, 128, 128, 1e4, 1), -1),
    ((A + 8, A, 1, 4, 2, 128, 128, 1e4, 1), -1),
    ((A, A, 1, 4, 2, 128, 127, 1e4, 1), -1),
    ((A, A, 1, 4, 2, 128, 130, 1e4, 1), -1),
    ((A, A, 1, 4, 2, 128, 0, 1e4, 1), -1),
    ((A, A, 1, 4, 2, 128, 128, 0.0, 1), -1),
    ((A, A, 1, 4, 2, 128, 128, float("inf"), 1), -1),
    ((A, A, 1, 4, 2, 96, 96, 1e4, 1), -2),
])
def test_rope_rejects_before_launch(L, args, status):
    assert L.swa_rope(*args, None) == status


@pytest.mark.parametrize("args,status", [
    ((None, A, A, A, A, A, A, 1, 8, 1, 128, 128, 128, 1e4, 1), -1),
    ((A, A, A, A, A, None, A, 1, 8, 1, 128, 128, 128, 1e4, 1), -1),
    ((A, A, A, A, A, A, A + 4, 1, 8, 1, 128, 128, 128, 1e4, 1), -1),
    ((A, A, A, A, A, A, A, 1, 8, 1, 128, 0, 128, 1e4, 1), -1),
    ((A, A, A, A, A, A, A, 1, 8, 1, 128, 128, 3, 1e4, 1), -1),
    ((A, A, A, A, A, A, A, 1, 8, 1, 128, 128, 128, -1.0, 1), -1),
    ((A, A, A, A, A, A, A, 1, 8, 1, 32, 128, 32, 1e4, 1), -2),
])
def test_rope_append_rejects_before_launch(L, args, status):
    assert L.swa_rope_append(*args, None) == status


def test_fwd_ex_rejects_before_launch(L):
    ok = (A, A, A, A, A, A, 1, 16, 8, 1, 128, 4, 1)
    assert L.swa_sink_fwd_ex(*ok, 7, None) == -1          # unknown output dtype
    assert L.swa_sink_fwd_ex(*ok[:4], None, *ok[5:], 1, None) == -1
    assert L.swa_sink_fwd_ex(*ok[:4], A + 8, *ok[5:], 1, None) == -1


def test_high_sparse_calls_reject_before_launch(L):
    # scores: null blockmax; topk: bad query block, capacity; sparse: bad QB
    assert L.swa_sink_fwd_scores(A, A, A, A, A, A, None, 1, 256, 8, 1, 128, 256, 1, 0, None) == -1
    assert L.swa_sink_fwd_scores(A, A, A, A, A, A, A, 1, 256, 4, 1, 128, 256, 1, 0, None) == -2
    assert L.swa_topk_blocks(A, A, 1, 1024, 2, 6, 4, None) == -1
    assert L.swa_topk_blocks(A, A, 1, 1024, 2, 256, 4, None) == -1
    assert L.swa_topk_blocks(A, A, 1, 1024, 2, 64, 0, None) == -1
    assert L.swa_topk_blocks(A, A, 1, 1024, 2, 64, 65, None) == -2
    assert L.swa_sink_sparse_fwd(A, A, A, A, A, A, A, 1, 1024, 8, 1, 128, 16, 4, 1, 0, None) == -2
    assert L.swa_sink_sparse_fwd(A, A, A, A, None, A, A, 1, 1024, 8, 1, 128, 64, 4, 1, 0,
                                 None) == -1


def test_fwd_host_rejects_before_launch(L):
    # q_h k_h v_h sink out_h lse_h | q_d k_d v_d out_d lse_d | B T Hq Hkv D W in out
    ok = (A, A, A, A, A, A, A, A, A, A, A, 2, 16, 8, 1, 128, 4, 1, 0)
    assert L.swa_sink_fwd_host(*ok[:4], None, *ok[5:], None) == -1        # no out_h
    assert L.swa_sink_fwd_host(*ok[:10], None, *ok[11:], None) == -1      # lse_h without lse_d
    assert L.swa_sink_fwd_host(*ok[:5], None, *ok[6:], None) == -1        # lse_d without lse_h
    assert L.swa_sink_fwd_host(*ok[:14], 3, *ok[15:], None) == -1         # Hq % Hkv != 0
    assert L.swa_sink_fwd_host(*ok[:17], 7, ok[18], None) == -1           # unknown input dtype
