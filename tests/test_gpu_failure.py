"""The failure path of a device-side wait, made to run out on purpose in the
permitted form: no fault, no trap, no unbounded spin.  One CTA of a small
sliding-window prefill issues none of its loads (swa_test_withhold_loads), so
its waits pass their 2 s limit.  The kernel must record a wait code in the
device error word, wind that CTA down (tensor memory freed, no copy left in
flight) and return; the other CTAs' tiles are complete, the device stays
usable, and the next call is bit-identical to one made before the fault."""
import pytest
import torch

import hybrid_sliding_window_02_b300 as swa
from hybrid_sliding_window_02_b300 import inputs as gen

pytestmark = pytest.mark.gpu

WAIT_CODES = set(range(0x101, 0x10d))   # kErrWait* in csrc/device_common.cuh


def _tiles_of_cta(cta, B, T, Hkv, sms):
    """(b, kvh, n) of the 16-position tiles CTA `cta` owns: persistent CTAs
    take contiguous ranges of tiles in (b, kv head, n) order."""
    nt = (T + 15) // 16
    total = B * Hkv * nt
    grid = min(total, sms)
    per, rem = divmod(total, grid)
    begin = cta * per + min(cta, rem)
    count = per + (1 if cta < rem else 0)
    out = []
    for u in range(begin, begin + count):
        bk, n = divmod(u, nt)
        b, kvh = divmod(bk, Hkv)
        out.append((b, kvh, n))
    return out


def test_withheld_loads_end_in_an_error_code_and_the_device_recovers(cuda_ok):
    B, T, Hq, Hkv, D, W = 1, 520, 64, 8, 128, 128
    dev = torch.device("cuda")
    assert swa.fwd_path(B, T, Hq, Hkv, D, W) == "tc_swa"
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=61, device=dev)
    assert swa.device_error() == 0
    ref_o, ref_l = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
    torch.cuda.synchronize()
    assert swa.device_error() == 0

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cta = 5
    out = torch.full((B, T, Hq, D), float("nan"), device=dev)
    lse = torch.full((B, Hq, T), float("nan"), device=dev)
    assert swa.lib().swa_test_withhold_loads(cta) == swa.SWA_OK
    swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, out, lse)
    code = swa.device_error()                # synchronises; ~2 s for the wait limit
    assert code in WAIT_CODES, hex(code)
    # the withholding CTA wrote nothing; every other row is the reference's
    own = torch.zeros(B, T, Hq, dtype=torch.bool, device=dev)
    for b, kvh, n in _tiles_of_cta(cta, B, T, Hkv, sms):
        own[b, 16 * n:16 * n + 16, 8 * kvh:8 * kvh + 8] = True
    assert own.any()
    assert torch.isnan(out[own]).all()
    assert torch.equal(out[~own], ref_o[~own])
    own_l = own.permute(0, 2, 1)
    assert torch.isnan(lse[own_l]).all()
    assert torch.equal(lse[~own_l], ref_l[~own_l])

    # the device is usable: the next calls are bit-identical and error-free
    for _ in range(2):
        o2, l2 = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W)
        torch.cuda.synchronize()
        assert torch.equal(o2, ref_o) and torch.equal(l2, ref_l)
    assert swa.device_error() == 0


def test_withhold_applies_to_one_launch_only(cuda_ok):
    # set and cancelled: the launch is normal
    x = gen.prefill_inputs(1, 64, 16, 2, 128, seed=62, device="cuda")
    assert swa.lib().swa_test_withhold_loads(0) == swa.SWA_OK
    assert swa.lib().swa_test_withhold_loads(-1) == swa.SWA_OK
    o, l = swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, 128)
    assert swa.device_error() == 0
    assert torch.isfinite(o).all() and torch.isfinite(l).all()
    assert swa.lib().swa_test_withhold_loads(-2) == swa.SWA_EINVAL
