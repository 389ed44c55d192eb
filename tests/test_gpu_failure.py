"""The decode kernel's failure path on the GPU, made to run without faulting
anything: a test-only launch issues no copy, so the kernel's bounded waits for
its staged cache rows (limited here to 1 ms) run out. The kernel must record
the wait timeout in the device error word, write nothing, and leave the context
usable for the next launch."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_05_b300 as swa
import swa_inputs
from parity import compare, scale_for

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT = 1  # the device error code of a wait that gave up


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


@pytest.mark.parametrize("B,Hq,Hkv,d,w,s,pos", [
    (64, 32, 8, 128, 64, 4, 1000),        # batch 64, no split
    (1, 32, 8, 128, 2048, 100, 5000),     # split over CTAs (workspace)
])
def test_stalled_decode_times_out_and_writes_nothing(B, Hq, Hkv, d, w, s, pos):
    dev = torch.device("cuda")
    sc = scale_for(d)
    swa.swa_device_error(clear=True)
    cache = swa.RingCache(B, Hkv, d, w, s, device=dev)
    _, k, v = swa_inputs.prefill_inputs(B, pos + 1, Hkv, Hkv, d, 7100 + pos)
    cache.append(k.to(dev), v.to(dev))
    posd = torch.full((B,), pos, dtype=torch.int32, device=dev)
    q = swa_inputs.decode_query(B, Hq, d, 7200).to(dev)
    sentinel = -3.5
    out = torch.full_like(q, sentinel)
    need = swa.swa_decode_workspace_size(B, Hq, Hkv, d, w, s)
    ws = torch.full((max(need, 16) // 4,), 7.0, dtype=torch.float32, device=dev) if need else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = swa.lib().swa_debug_decode_timeout(
        _p(q), _p(cache.k), _p(cache.v), _p(posd), _p(out), B, Hq, Hkv, d, w, s,
        ctypes.c_float(sc), _p(ws), need, ctypes.c_ulonglong(1_000_000), 1, stream)
    assert rc == swa.SWA_OK, swa.swa_last_error()
    torch.cuda.synchronize()
    assert swa.swa_device_error(clear=True) == WAIT_TIMEOUT
    assert torch.all(out == sentinel), "a timed-out decode wrote its output"
    if ws is not None:
        assert torch.all(ws == 7.0), "a timed-out decode wrote its workspace"
    # the context is still usable: the same decode, not stalled, is correct
    res = swa.swa_decode(q, cache.k, cache.v, posd, w, s, sc)
    torch.cuda.synchronize()
    assert swa.swa_device_error(clear=True) == 0
    keys = oracle.keyset(pos, w, s)
    want = np.stack([oracle.decode(q[b].cpu(), keys, k[b, keys], v[b, keys], pos, w, s, sc)[0]
                     for b in range(B)])
    compare(res.cpu(), want, "decode after the timed-out launch")


def test_unstalled_debug_launch_matches_decode():
    """The test-only entry point with stall = 0 is the ordinary decode."""
    B, Hq, Hkv, d, w, s, pos = 4, 8, 2, 64, 40, 4, 300
    dev = torch.device("cuda")
    sc = scale_for(d)
    cache = swa.RingCache(B, Hkv, d, w, s, device=dev)
    _, k, v = swa_inputs.prefill_inputs(B, pos + 1, Hkv, Hkv, d, 7300)
    cache.append(k.to(dev), v.to(dev))
    posd = torch.full((B,), pos, dtype=torch.int32, device=dev)
    q = swa_inputs.decode_query(B, Hq, d, 7400).to(dev)
    out = torch.empty_like(q)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = swa.lib().swa_debug_decode_timeout(
        _p(q), _p(cache.k), _p(cache.v), _p(posd), _p(out), B, Hq, Hkv, d, w, s,
        ctypes.c_float(sc), None, 0, ctypes.c_ulonglong(2_000_000_000), 0, stream)
    assert rc == swa.SWA_OK
    ref = swa.swa_decode(q, cache.k, cache.v, posd, w, s, sc)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert swa.swa_device_error(clear=True) == 0
