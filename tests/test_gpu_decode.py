"""Ring-cache append and SWA(w, s) decode on the GPU (through the C ABI)
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_05_b300 as swa
import swa_inputs
from parity import compare, prefill_case, sample_rows, scale_for

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(autouse=True)
def _device_error_clean():
    swa.swa_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert swa.swa_device_error(clear=True) == 0


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16)


@pytest.mark.parametrize("w,s", [(7, 3), (4, 0), (1, 2), (64, 4)])
def test_append_slots_bitexact(w, s):
    """After every append call, slot i of the cache holds exactly the K/V row
    of the position the oracle's circular buffer puts there."""
    B, Hkv, d = 2, 3, 64
    total = 3 * (s + w) + 40
    _, k, v = prefill_case(B, total, Hkv, Hkv, d, 4001)
    cache = swa.RingCache(B, Hkv, d, w, s)
    rng = np.random.default_rng(w * 10 + s)
    pos = 0
    while pos < total:
        T = int(min(total - pos, rng.choice([1, 2, 3, 5, w + 1, 2 * w + s + 3])))
        cache.append(k[:, pos:pos + T].cuda(), v[:, pos:pos + T].cuda())
        pos += T
        torch.cuda.synchronize()
        slots = oracle.ring_contents(pos - 1, w, s)
        kc, vc = _bits(cache.k), _bits(cache.v)
        kb, vb = _bits(k), _bits(v)
        for i, p in enumerate(slots.tolist()):
            if p >= 0:
                assert torch.equal(kc[:, :, i], kb[:, p]), (pos, i, p)
                assert torch.equal(vc[:, :, i], vb[:, p]), (pos, i, p)


@pytest.mark.parametrize("case", [
    # B, L, Hq, Hkv, d, w, s
    (1, 256, 4, 1, 64, 64, 4),
    (2, 150, 32, 8, 128, 16, 4),
    (1, 120, 6, 2, 64, 9, 0),
    (1, 100, 8, 8, 128, 20, 30),
    (2, 90, 16, 2, 64, 200, 4),
], ids=lambda c: "B%d_L%d_Hq%d_Hkv%d_d%d_w%d_s%d" % c)
def test_decode_equals_prefill_rows(case):
    """Token-by-token append + decode reproduces the prefill row at every
    position (both sides checked against the oracle)."""
    B, L, Hq, Hkv, d, w, s = case
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 4100 + L, sink_rows=min(s, L))
    sc = scale_for(d)
    ref, _ = oracle.prefill(q, k, v, w, s, sc)
    cache = swa.RingCache(B, Hkv, d, w, s)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    outs = []
    for t in range(L):
        cache.append(kd[:, t:t + 1].contiguous(), vd[:, t:t + 1].contiguous())
        outs.append(cache.decode(qd[:, t].contiguous(), sc))
    dec = torch.stack(outs, dim=1)
    compare(dec.cpu(), ref, "decode")
    pre = swa.swa_prefill(qd, kd, vd, w, s, sc)
    torch.cuda.synchronize()
    compare(pre.cpu(), ref, "prefill")


def _keyed(seed, stream, B, Hkv, positions, d):
    rows = [[swa_inputs.keyed_rows(seed, stream, b, h, positions, d) for h in range(Hkv)]
            for b in range(B)]
    # -> [B, T, Hkv, d]
    return torch.stack([torch.stack(r, dim=1) for r in rows], dim=0)


@pytest.mark.parametrize("P", [128, 1024, 16384, 262143])
def test_batch64_decode_positions(P):
    """Batch 64, Hq=32, Hkv=8, d=128, SWA(64, 4), 68-slot cache: the cache is
    fast-forwarded to position P with the position-keyed generator, then three
    single-token steps P+1..P+3 are appended and decoded."""
    B, Hq, Hkv, d, w, s = 64, 32, 8, 128, 64, 4
    seed = 1003
    sc = scale_for(d)
    cache = swa.RingCache(B, Hkv, d, w, s)
    sinks = np.arange(s)
    cache.append(_keyed(seed, 0, B, Hkv, sinks, d).cuda(), _keyed(seed, 1, B, Hkv, sinks, d).cuda())
    lo = max(s, P - w + 1)
    win = np.arange(lo, P + 1)
    # jump: the window part starts at lo, not at s
    cache.seek(lo)
    cache.append(_keyed(seed, 0, B, Hkv, win, d).cuda(), _keyed(seed, 1, B, Hkv, win, d).cuda())
    for step in range(1, 4):
        pos = P + step
        kn = _keyed(seed, 0, B, Hkv, [pos], d)
        vn = _keyed(seed, 1, B, Hkv, [pos], d)
        cache.append(kn.cuda(), vn.cuda())
        qn = swa_inputs.decode_query(B, Hq, d, seed * 1000 + pos)
        out = cache.decode(qn.cuda(), sc).cpu()
        keys = oracle.keyset(pos, w, s)
        assert len(keys) == s + w
        ref = np.zeros((B, Hq, d))
        for b in range(B):
            hk = torch.stack([swa_inputs.keyed_rows(seed, 0, b, h, keys, d) for h in range(Hkv)], 1)
            hv = torch.stack([swa_inputs.keyed_rows(seed, 1, b, h, keys, d) for h in range(Hkv)], 1)
            ref[b], _ = oracle.decode(qn[b], keys, hk, hv, pos, w, s, sc)
        compare(out, ref, f"P={P} step {step}")


@pytest.mark.parametrize("w,s,pos", [(2048, 100, 5000), (2048, 100, 1000), (16640, 0, 16383),
                                     (300, 4, 299)])
def test_split_kv_decode(w, s, pos):
    """One sequence over a long cache: the split-KV path with LSE combine."""
    B, Hq, Hkv, d = 1, 32, 8, 128
    assert swa.swa_decode_workspace_size(B, Hq, Hkv, d, w, s) > 0
    L = pos + 1
    _, k, v = prefill_case(B, L, Hkv, Hkv, d, 4200 + pos)
    q = swa_inputs.decode_query(B, Hq, d, 4300 + pos)
    cache = swa.RingCache(B, Hkv, d, w, s)
    cache.append(k.cuda(), v.cuda())
    out = cache.decode(q.cuda()).cpu()
    keys = oracle.keyset(pos, w, s)
    ref, _ = oracle.decode(q[0], keys, k[0, keys], v[0, keys], pos, w, s, scale_for(d))
    compare(out[0], ref, f"split w={w} s={s} pos={pos}")


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 4, 64), (6, 2, 128), (16, 2, 64), (32, 4, 128),
                                      (12, 1, 128)])
def test_decode_group_sizes(Hq, Hkv, d):
    B, w, s, pos = 5, 24, 3, 70
    _, k, v = prefill_case(B, pos + 1, Hkv, Hkv, d, 4400 + Hq)
    q = swa_inputs.decode_query(B, Hq, d, 4500 + Hq)
    cache = swa.RingCache(B, Hkv, d, w, s)
    cache.append(k.cuda(), v.cuda())
    out = cache.decode(q.cuda()).cpu()
    keys = oracle.keyset(pos, w, s)
    ref = np.stack([oracle.decode(q[b], keys, k[b, keys], v[b, keys], pos, w, s, scale_for(d))[0]
                    for b in range(B)])
    compare(out, ref, f"G={Hq // Hkv}")


def test_hybrid_stack_prefill_then_decode():
    """8 layers alternating SWA(2048, 100) and full causal, B=1, L=16384,
    Hq=32, Hkv=8, d=128, through the package's HybridStack driver: fresh seeded
    q/k/v per layer, prefill, then 256 decode steps through all layers (step by
    step, as a decoder runs). Sampled prefill rows and decode steps of every
    layer are checked against the oracle."""
    B, L, Hq, Hkv, d, steps = 1, 16384, 32, 8, 128, 256
    sc = scale_for(d)
    check_steps = {0, 1, 127, 255}
    windows = swa.hybrid_layer_windows(8, L, steps)
    assert windows[0] == (2048, 100) and windows[1] == (L + steps, 0)
    host, toks = [], []
    for layer in range(8):
        seed = 1000 + 5 * 100 + layer
        q, k, v = prefill_case(B, L, Hq, Hkv, d, seed)
        g = torch.Generator("cpu").manual_seed(seed + 77)
        qs = torch.randn(steps, B, Hq, d, generator=g).to(torch.bfloat16)
        ks = torch.randn(steps, B, 1, Hkv, d, generator=g).to(torch.bfloat16)
        vs = torch.randn(steps, B, 1, Hkv, d, generator=g).to(torch.bfloat16)
        host.append((q, k, v, qs, ks, vs))
        toks.append((qs.cuda(), ks[:, :, 0].cuda(), vs[:, :, 0].cuda()))
    stack = swa.HybridStack(B, Hq, Hkv, d, windows, scale=sc)
    outs = stack.prefill([(q.cuda(), k.cuda(), v.cuda()) for q, k, v, *_ in host])
    dec = {}
    for i in range(steps):
        o = stack.step([(qs[i], ks[i], vs[i]) for qs, ks, vs in toks])
        if i in check_steps:
            dec[i] = [x.clone() for x in o]
    torch.cuda.synchronize()
    for layer, ((w, s), (q, k, v, qs, ks, vs)) in enumerate(zip(windows, host)):
        # SWA layers: every row t < w + s + 128; full layers: the first 512;
        # both: the last 128 rows and 512 random ones
        rows = sample_rows(L, w, s, 512, seed=layer, head_cap=512 if w >= L else None)
        ref, _ = oracle.prefill(q, k, v, w, s, sc, rows=rows)
        compare(outs[layer][:, torch.from_numpy(rows).cuda()].cpu(), ref, f"layer {layer} prefill")
        hist_k = torch.cat([k[0], ks[:, 0, 0]], 0)
        hist_v = torch.cat([v[0], vs[:, 0, 0]], 0)
        for i in sorted(check_steps):
            pos = L + i
            keys = oracle.keyset(pos, w, s)
            r, _ = oracle.decode(qs[i, 0], keys, hist_k[keys], hist_v[keys], pos, w, s, sc)
            compare(dec[i][layer][0].cpu(), r, f"layer {layer} decode step {i}")


@pytest.mark.parametrize("case", [
    # B, L, Hq, Hkv, d, w, s
    (1, 256, 4, 1, 64, 64, 4),
    (2, 150, 32, 8, 128, 16, 4),
    (1, 120, 6, 2, 64, 9, 0),
    (2, 90, 16, 2, 64, 200, 4),
], ids=lambda c: "B%d_L%d_Hq%d_Hkv%d_d%d_w%d_s%d" % c)
def test_append_decode_equals_prefill_rows(case):
    """swa_append_decode (append the token, then decode it, in one launch)
    reproduces every prefill row, and leaves the cache bit-identical to
    swa_cache_append."""
    B, L, Hq, Hkv, d, w, s = case
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 4700 + L, sink_rows=min(s, L))
    sc = scale_for(d)
    ref, _ = oracle.prefill(q, k, v, w, s, sc)
    fused = swa.RingCache(B, Hkv, d, w, s)
    plain = swa.RingCache(B, Hkv, d, w, s)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    outs = []
    for t in range(L):
        outs.append(fused.step(qd[:, t].contiguous(), kd[:, t].contiguous(), vd[:, t].contiguous(), sc))
        plain.append(kd[:, t:t + 1].contiguous(), vd[:, t:t + 1].contiguous())
    dec = torch.stack(outs, dim=1)
    torch.cuda.synchronize()
    compare(dec.cpu(), ref, "append_decode")
    assert torch.equal(_bits(fused.k), _bits(plain.k)) and torch.equal(_bits(fused.v), _bits(plain.v))


@pytest.mark.parametrize("w,s,pos", [(2048, 100, 5000), (16640, 0, 9000)])
def test_append_decode_split_kv(w, s, pos):
    """The fused call on the split-KV path (one sequence, long cache)."""
    B, Hq, Hkv, d = 1, 32, 8, 128
    _, k, v = prefill_case(B, pos + 1, Hkv, Hkv, d, 4800 + pos)
    q = swa_inputs.decode_query(B, Hq, d, 4900 + pos)
    cache = swa.RingCache(B, Hkv, d, w, s)
    cache.append(k[:, :pos].cuda(), v[:, :pos].cuda())
    out = cache.step(q.cuda(), k[:, pos].contiguous().cuda(), v[:, pos].contiguous().cuda()).cpu()
    keys = oracle.keyset(pos, w, s)
    ref, _ = oracle.decode(q[0], keys, k[0, keys], v[0, keys], pos, w, s, scale_for(d))
    compare(out[0], ref, f"fused split w={w} s={s} pos={pos}")
