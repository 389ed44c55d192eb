"""swa_decode_noalloc, the decode entry point that allocates nothing.

Some callers cannot allocate device memory when they call decode: a serving
engine that owns all device memory in a fixed pool and forbids allocation
inside a step (cudaMalloc can synchronise the device and can fail under memory
pressure), or plain C code with no allocator for scratch buffers. For them
swa_decode_noalloc keeps the split-KV partial results in a fixed scratch array
compiled into libswa.so instead of a caller workspace.

These tests call it through the C ABI and check its output against swa_decode
(the entry point that takes a workspace) and against the fp64 oracle, on two
calls in a row, so that the scratch left over from the first call cannot leak
into the second.
This file is collected last on purpose: a run that stops at the first failure
has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_05_b300 as swa
import swa_inputs
from parity import MAX_ABS, REL_L2, compare

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(q, kc, vc, pos, out, w, s, scale):
    B, Hq, d = q.shape
    Hkv = kc.shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return swa.lib().swa_decode_noalloc(_p(q), _p(kc), _p(vc), _p(pos), _p(out), B, Hq, Hkv, d,
                                        w, s, ctypes.c_float(scale), stream)


def _close(got, ref, what):
    g = got.float().cpu().double().numpy()
    r = ref.float().cpu().double().numpy()
    err = g - r
    ma = float(np.abs(err).max())
    rl = float(np.linalg.norm(err) / np.linalg.norm(r))
    assert np.all(np.isfinite(g)), what
    assert ma <= MAX_ABS and rl <= REL_L2, f"{what}: max-abs {ma:.3e} rel-L2 {rl:.3e}"


@pytest.mark.parametrize("B,Hq,Hkv,d,w,s,pos,split", [
    (1, 32, 8, 128, 2048, 100, 5000, True),    # one long sequence: split-KV, uses the scratch
    (1, 32, 8, 128, 8192, 0, 9000, True),      # long window, 64 splits of 128 slots
    (3, 12, 4, 64, 300, 4, 700, True),         # group of 3, d = 64
    (64, 32, 8, 128, 64, 4, 1000, False),      # batch 64: no split, no scratch needed
])
def test_noalloc_decode_matches_workspace_decode(B, Hq, Hkv, d, w, s, pos, split):
    need = swa.swa_decode_workspace_size(B, Hq, Hkv, d, w, s)
    assert (need > 0) == split
    assert need <= 2 << 20
    dev = torch.device("cuda")
    scale = 1.0 / np.sqrt(d)
    cache = swa.RingCache(B, Hkv, d, w, s, device=dev)
    _, k, v = swa_inputs.prefill_inputs(B, pos + 1, Hkv, Hkv, d, 9100 + pos)
    cache.append(k.to(dev), v.to(dev))
    posd = torch.full((B,), pos, dtype=torch.int32, device=dev)
    for call in range(2):
        q = swa_inputs.decode_query(B, Hq, d, 9200 + 10 * pos + call).to(dev)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev) if need else None
        ref = swa.swa_decode(q, cache.k, cache.v, posd, w, s, scale, workspace=ws)
        got = torch.full_like(q, float("nan"))
        assert _noalloc(q, cache.k, cache.v, posd, got, w, s, scale) == swa.SWA_OK, swa.swa_last_error()
        torch.cuda.synchronize()
        _close(got, ref, f"call {call}")
        keys = oracle.keyset(pos, w, s)
        want = np.stack([oracle.decode(q[b].cpu(), keys, k[b, keys], v[b, keys], pos, w, s,
                                       scale)[0] for b in range(B)])
        compare(got.cpu(), want, f"call {call} vs oracle")
    assert swa.swa_device_error(clear=True) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # B=2, Hq=1024, Hkv=8, d=128: the split-KV partials need more than 2 MiB
    B, Hq, Hkv, d, w, s = 2, 1024, 8, 128, 4096, 0
    assert swa.swa_decode_workspace_size(B, Hq, Hkv, d, w, s) > (2 << 20)
    dummy = ctypes.c_void_p(4096)
    rc = swa.lib().swa_decode_noalloc(dummy, dummy, dummy, dummy, dummy, B, Hq, Hkv, d, w, s,
                                      ctypes.c_float(0.1), None)
    assert rc == swa.SWA_ERR_UNSUPPORTED
    assert "maximum" in swa.swa_last_error()
