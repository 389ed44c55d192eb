"""The SWAA "FA decode" mode on the GPU against the fp64 oracle: the prompt is
prefilled with SWA(w, s) (row t attends to K(t) of SWA(w, s)), every position
is kept, and each decoded token attends to the whole history with full causal
attention (position p attends to K(p) of SWA(inf, 0) = 0 .. p)."""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_05_b300 as swa
from parity import MAX_ABS, REL_L2, compare, prefill_case, sample_rows, scale_for

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _device_error_clean():
    swa.swa_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert swa.swa_device_error(clear=True) == 0


def _tokens(seed, steps, B, Hq, Hkv, d):
    g = torch.Generator("cpu").manual_seed(seed)
    qs = torch.randn(steps, B, Hq, d, generator=g).to(torch.bfloat16)
    ks = torch.randn(steps, B, Hkv, d, generator=g).to(torch.bfloat16)
    vs = torch.randn(steps, B, Hkv, d, generator=g).to(torch.bfloat16)
    return qs, ks, vs


def _differs(a, b):
    """a and b are further apart than the parity tolerance (so the test tells
    full-attention decode from sliding-window decode)."""
    err = a - b
    return (np.max(np.abs(err)) > MAX_ABS or
            np.linalg.norm(err) / np.linalg.norm(b) > REL_L2)


def _run(B, L, Hq, Hkv, d, w, s, steps, seed, rows, check_steps):
    sc = scale_for(d)
    q, k, v = prefill_case(B, L, Hq, Hkv, d, seed, sink_rows=min(s, 4))
    qs, ks, vs = _tokens(seed + 1, steps, B, Hq, Hkv, d)
    layer = swa.AttentionLayer(B, Hq, Hkv, d, w, s, scale=sc, fa_decode=True, max_len=L + steps)
    assert (layer.cache_w, layer.cache_s) == (L + steps, 0)
    out = layer.prefill(q.cuda(), k.cuda(), v.cuda())
    dec = {}
    for i in range(steps):
        o = layer.step(qs[i].cuda(), ks[i].cuda(), vs[i].cuda())
        if i in check_steps:
            dec[i] = o.clone()
    torch.cuda.synchronize()
    # prefill rows: SWA(w, s)
    ref, _ = oracle.prefill(q, k, v, w, s, sc, rows=rows)
    compare(out[:, torch.from_numpy(rows).cuda()].cpu(), ref, "FA-decode layer prefill")
    # decode rows: full causal over the prompt and every decoded token
    hist_k = torch.cat([k, ks.permute(1, 0, 2, 3)], 1)     # [B, L + steps, Hkv, d]
    hist_v = torch.cat([v, vs.permute(1, 0, 2, 3)], 1)
    for i in sorted(check_steps):
        pos = L + i
        full = oracle.keyset(pos, pos + 1, 0)
        assert len(full) == pos + 1
        swa_keys = oracle.keyset(pos, w, s)
        want = np.stack([oracle.decode(qs[i, b], full, hist_k[b, full], hist_v[b, full], pos,
                                       pos + 1, 0, sc)[0] for b in range(B)])
        got = dec[i].cpu()
        compare(got, want, f"FA decode step {i}")
        sliding = np.stack([oracle.decode(qs[i, b], swa_keys, hist_k[b, swa_keys],
                                          hist_v[b, swa_keys], pos, w, s, sc)[0]
                            for b in range(B)])
        assert _differs(want, sliding), "full and sliding-window decode agree: test too weak"


def test_fa_decode_small_every_row_and_step():
    """B=2, L=300, Hq=8, Hkv=2, d=64, SWA(32, 4) prefill, 40 full-attention
    decode steps: every prefill row and every decode step."""
    B, L, Hq, Hkv, d, w, s, steps = 2, 300, 8, 2, 64, 32, 4, 40
    _run(B, L, Hq, Hkv, d, w, s, steps, 6100, np.arange(L), set(range(steps)))


def test_fa_decode_swaa_layer():
    """The SWAA setting: B=1, L=16384, Hq=32, Hkv=8, d=128, SWA(2048, 100)
    prefill, then 64 full-attention decode steps over the whole history."""
    B, L, Hq, Hkv, d, w, s, steps = 1, 16384, 32, 8, 128, 2048, 100, 64
    rows = sample_rows(L, w, s, 1024, seed=61)
    _run(B, L, Hq, Hkv, d, w, s, steps, 6200, rows, {0, 1, 31, 63})


def test_fa_decode_hybrid_stack():
    """A 4-layer SWAA stack (SWA(2048, 100) layers in FA-decode mode between
    full-causal layers), B=1, L=4096: every layer's decode is full attention."""
    B, L, Hq, Hkv, d, steps = 1, 4096, 32, 8, 128, 8
    sc = scale_for(d)
    windows = swa.hybrid_layer_windows(4, L, steps)
    stack = swa.HybridStack(B, Hq, Hkv, d, windows, scale=sc, fa_decode=True, max_len=L + steps)
    assert [l.fa_decode for l in stack.layers] == [True, False, True, False]
    assert all((l.cache_w, l.cache_s) == (L + steps, 0) for l in stack.layers)
    host = [prefill_case(B, L, Hq, Hkv, d, 6300 + i) for i in range(4)]
    toks = [_tokens(6400 + i, steps, B, Hq, Hkv, d) for i in range(4)]
    stack.prefill([(q.cuda(), k.cuda(), v.cuda()) for q, k, v in host])
    last = None
    for i in range(steps):
        last = stack.step([(qs[i].cuda(), ks[i].cuda(), vs[i].cuda()) for qs, ks, vs in toks])
    torch.cuda.synchronize()
    pos = L + steps - 1
    for layer, ((q, k, v), (qs, ks, vs)) in enumerate(zip(host, toks)):
        hk = torch.cat([k[0], ks[:, 0]], 0)
        hv = torch.cat([v[0], vs[:, 0]], 0)
        full = np.arange(pos + 1)
        want, _ = oracle.decode(qs[-1, 0], full, hk, hv, pos, pos + 1, 0, sc)
        compare(last[layer][0].cpu(), want, f"stack layer {layer}")
