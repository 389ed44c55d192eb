"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

Each ``check_*`` takes a loaded oracle library (the real one, or a deliberately
broken copy in the mutation test) and raises AssertionError when the oracle
disagrees with the pin. None of them re-types the oracle's own formula: the
references are the page's boolean-mask definition, closed forms, a library
routine (torch's fp64 scaled_dot_product_attention), exact special cases, and
the page's worked examples in tests/golden/.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
import swa_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "pages_examples.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def count_closed_form(t: int, w: int, s: int) -> int:
    """|K(t)|: min(t+1, w) window keys plus the sinks left of the window."""
    return min(t + 1, w) + min(s, max(0, t - w + 1))


def _sdpa_reference(q, k, v, w, s, scale):
    """torch fp64 SDPA with the page's boolean mask (clamped to causal) and
    K/V heads repeated for GQA. q [B,L,Hq,d] bf16 -> out [B,L,Hq,d] float64."""
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    qd = q.double().permute(0, 2, 1, 3)
    kd = k.double().repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    vd = v.double().repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    mask = torch.from_numpy(oracle.swa_mask(L, w, s) & np.tril(np.ones((L, L), dtype=bool)))
    o = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask, scale=float(np.float32(scale)))
    return o.permute(0, 2, 1, 3).numpy()


# ---------------------------------------------------------------- key sets

def check_keymask_vs_pseudocode(lib, Lmax=20):
    for L in range(1, Lmax + 1):
        tril = np.tril(np.ones((L, L), dtype=bool))
        for w in range(1, L + 3):
            for s in range(0, L + 3):
                got = oracle.keymask(L, w, s, lib=lib)
                want = oracle.swa_mask(L, w, s) & tril
                assert np.array_equal(got, want), (L, w, s)


def check_counts_closed_form(lib):
    for (L, w, s) in [(64, 1, 0), (64, 5, 3), (200, 64, 4), (300, 17, 40), (90, 100, 4)]:
        for t in range(L):
            n = len(oracle.keyset(t, w, s, lib=lib))
            assert n == count_closed_form(t, w, s), (L, w, s, t, n)
    # per-head in-band pair totals of the tiny and the Llama-shaped prefill
    for (L, w, s, total) in [(256, 64, 4, 15130), (4096, 128, 4, 532026)]:
        got = sum(len(oracle.keyset(t, w, s, lib=lib)) for t in range(L))
        assert got == total, (L, w, s, got)


def check_full_window_is_causal(lib):
    for L in (1, 7, 33):
        for w in (L, L + 1, 5 * L):
            for s in (0, 3, L + 2):
                assert np.array_equal(oracle.keymask(L, w, s, lib=lib),
                                      np.tril(np.ones((L, L), dtype=bool))), (L, w, s)


def check_no_sinks_is_band(lib):
    # x_t equation: i runs over max(1, t-w+1) .. t in 1-indexed positions
    for L in (9, 40):
        for w in (1, 2, 5, 39, 40, 41):
            want = np.zeros((L, L), dtype=bool)
            for t1 in range(1, L + 1):
                for i1 in range(max(1, t1 - w + 1), t1 + 1):
                    want[t1 - 1, i1 - 1] = True
            assert np.array_equal(oracle.keymask(L, w, 0, lib=lib), want), (L, w)


# ---------------------------------------------------------------- values

def check_prefill_vs_sdpa(lib):
    cases = [
        # B, L, Hq, Hkv, d, w, s, seed, sink_rows
        (2, 48, 4, 2, 16, 5, 3, 11, 3),
        (1, 40, 2, 1, 8, 1, 0, 12, 0),
        (1, 37, 3, 3, 8, 8, 0, 13, 0),
        (2, 33, 4, 1, 16, 64, 4, 14, 4),   # w >= L
        (1, 50, 2, 2, 8, 7, 60, 15, 0),    # s > L
        (1, 64, 8, 2, 32, 16, 4, 16, 4),
    ]
    for (B, L, Hq, Hkv, d, w, s, seed, sr) in cases:
        q, k, v = swa_inputs.prefill_inputs(B, L, Hq, Hkv, d, seed, sink_rows=sr)
        scale = 1.0 / math.sqrt(d)
        out, _ = oracle.prefill(q, k, v, w, s, scale, lib=lib)
        ref = _sdpa_reference(q, k, v, w, s, scale)
        err = np.max(np.abs(out - ref))
        assert err < 1e-12, (B, L, Hq, Hkv, d, w, s, err)


def check_large_logits(lib):
    # scores of magnitude ~1e3: exp() without the max shift overflows
    q, k, v = swa_inputs.prefill_inputs(1, 24, 2, 1, 16, 21)
    q = (q.float() * 64).to(torch.bfloat16)
    out, _ = oracle.prefill(q, k, v, 6, 2, 1.0, lib=lib)
    ref = _sdpa_reference(q, k, v, 6, 2, 1.0)
    assert np.all(np.isfinite(out))
    assert np.max(np.abs(out - ref)) < 1e-9


def check_full_causal_vs_sdpa_is_causal(lib):
    B, L, Hq, Hkv, d = 1, 45, 4, 2, 16
    q, k, v = swa_inputs.prefill_inputs(B, L, Hq, Hkv, d, 31)
    scale = 0.3
    out, _ = oracle.prefill(q, k, v, L + 7, 0, scale, lib=lib)
    G = Hq // Hkv
    o = F.scaled_dot_product_attention(
        q.double().permute(0, 2, 1, 3),
        k.double().repeat_interleave(G, dim=2).permute(0, 2, 1, 3),
        v.double().repeat_interleave(G, dim=2).permute(0, 2, 1, 3),
        is_causal=True, scale=float(np.float32(scale))).permute(0, 2, 1, 3).numpy()
    assert np.max(np.abs(out - o)) < 1e-12


def check_window_one_identity(lib):
    q, k, v = swa_inputs.prefill_inputs(2, 30, 4, 2, 8, 41)
    out, _ = oracle.prefill(q, k, v, 1, 0, 0.125, lib=lib)
    want = v.double().repeat_interleave(2, dim=2).numpy()
    assert np.array_equal(out, want)


def check_zero_query_mean(lib):
    B, L, Hq, Hkv, d, w, s = 1, 40, 2, 1, 8, 6, 3
    _, k, v = swa_inputs.prefill_inputs(B, L, Hq, Hkv, d, 51)
    q = torch.zeros(B, L, Hq, d, dtype=torch.bfloat16)
    out, _ = oracle.prefill(q, k, v, w, s, 0.35, lib=lib)
    vd = v.double().numpy()
    mask = oracle.swa_mask(L, w, s) & np.tril(np.ones((L, L), dtype=bool))
    for t in range(L):
        mean = vd[0, mask[t], 0, :].mean(axis=0)
        for h in range(Hq):
            assert np.max(np.abs(out[0, t, h] - mean)) < 1e-13, t


def check_constant_values(lib):
    q, k, _ = swa_inputs.prefill_inputs(1, 36, 4, 2, 16, 61, sink_rows=4)
    v = torch.full((1, 36, 2, 16), 0.8125, dtype=torch.bfloat16)
    out, _ = oracle.prefill(q, k, v, 5, 4, 0.25, lib=lib)
    assert np.max(np.abs(out - 0.8125)) < 1e-14


def check_gqa_equals_repeated_mha(lib):
    q, k, v = swa_inputs.prefill_inputs(2, 29, 6, 2, 8, 71, sink_rows=2)
    a, la = oracle.prefill(q, k, v, 4, 2, 0.5, lib=lib)
    b, lb = oracle.prefill(q, k.repeat_interleave(3, dim=2), v.repeat_interleave(3, dim=2),
                           4, 2, 0.5, lib=lib)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def check_weights_sum_to_one(lib):
    q, k, v = swa_inputs.prefill_inputs(1, 40, 2, 1, 16, 81, sink_rows=4)
    for t in range(40):
        wts = oracle.weights(q, k, 6, 4, 0.25, 0, 1, t, lib=lib)
        assert len(wts) == count_closed_form(t, 6, 4)
        assert abs(wts.sum() - 1.0) < 1e-15 * max(1, len(wts)) * 4
        assert np.all(wts > 0)


def check_weights_vs_torch_softmax(lib):
    """Each row's weights equal torch's fp64 softmax (a library routine) of the
    scaled scores q_t . k_j over the page's boolean mask row (clamped to
    causal), with the query head reading KV head hq // (Hq / Hkv). The
    configuration has a group of 3 query heads per KV head (so hq // G and
    hq % Hkv differ for most heads) and a scale far from 1."""
    B, L, Hq, Hkv, d, w, s, scale = 2, 33, 6, 2, 16, 5, 3, 0.37
    q, k, _ = swa_inputs.prefill_inputs(B, L, Hq, Hkv, d, 83, sink_rows=3)
    G = Hq // Hkv
    kd = k.double().repeat_interleave(G, dim=2)          # [B, L, Hq, d]: head hq reads hq // G
    mask = torch.from_numpy(oracle.swa_mask(L, w, s) & np.tril(np.ones((L, L), dtype=bool)))
    sc = float(np.float32(scale))
    for b in range(B):
        for hq in range(Hq):
            x = (q.double()[b, :, hq, :] @ kd[b, :, hq, :].T) * sc       # [L, L]
            x = x.masked_fill(~mask, -math.inf)
            p = torch.softmax(x, dim=1).numpy()
            for t in range(L):
                want = p[t][mask[t].numpy()]
                got = oracle.weights(q, k, w, s, scale, b, hq, t, lib=lib)
                assert got.shape == want.shape, (b, hq, t)
                assert np.max(np.abs(got - want)) < 1e-13, (b, hq, t)


def check_lse_vs_logsumexp(lib):
    q, k, v = swa_inputs.prefill_inputs(1, 30, 2, 2, 16, 91, sink_rows=2)
    w, s, scale = 7, 2, 0.25
    _, lse = oracle.prefill(q, k, v, w, s, scale, lib=lib)
    mask = oracle.swa_mask(30, w, s) & np.tril(np.ones((30, 30), dtype=bool))
    qd, kd = q.double(), k.double()
    for h in range(2):
        sc = (qd[0, :, h, :] @ kd[0, :, h, :].T) * float(np.float32(scale))
        sc[~torch.from_numpy(mask)] = -math.inf
        ref = torch.logsumexp(sc, dim=1).numpy()
        assert np.max(np.abs(lse[0, :, h] - ref)) < 1e-12


# ---------------------------------------------------------------- decode and ring

def check_decode_equals_prefill_row(lib):
    B, L, Hq, Hkv, d, w, s = 1, 48, 4, 2, 16, 6, 3
    q, k, v = swa_inputs.prefill_inputs(B, L, Hq, Hkv, d, 101, sink_rows=3)
    scale = 0.25
    out, lse = oracle.prefill(q, k, v, w, s, scale, lib=lib)
    for pos in range(L):
        hist = np.arange(pos + 1)
        o, l = oracle.decode(q[0, pos], hist, k[0, :pos + 1], v[0, :pos + 1], pos, w, s, scale, lib=lib)
        assert np.max(np.abs(o - out[0, pos])) < 1e-12, pos
        assert np.max(np.abs(l - lse[0, pos])) < 1e-12, pos
        # the ring contents alone are a sufficient history
        slots = oracle.ring_contents(pos, w, s, lib=lib)
        held = slots[slots >= 0]
        o2, _ = oracle.decode(q[0, pos], held, k[0, held], v[0, held], pos, w, s, scale, lib=lib)
        assert np.max(np.abs(o2 - out[0, pos])) < 1e-12, pos


def check_ring_page_example(lib):
    g = golden()["ring_eviction"]
    slots = oracle.ring_contents(g["tokens_appended"] - 1, g["w"], g["s"], lib=lib)
    assert sorted(slots.tolist()) == g["held_positions"]
    for p in g["evicted_positions"]:
        assert p not in slots.tolist()


def check_ring_holds_keyset(lib):
    for w in (1, 2, 3, 4, 7, 64):
        for s in (0, 1, 4, 5):
            for last in list(range(0, 3 * (s + w) + 6)) + [65536, 262143]:
                slots = oracle.ring_contents(last, w, s, lib=lib)
                held = sorted(int(p) for p in slots if p >= 0)
                assert held == oracle.keyset(last, w, s, lib=lib).tolist(), (w, s, last)
                assert len(set(held)) == len(held)


def check_footprint(lib):
    g = golden()["sink_window_footprint"]
    slots = oracle.ring_contents(g["context"] - 1, g["w"], g["s"], lib=lib)
    assert int((slots >= 0).sum()) == g["held_tokens"]
    assert len(oracle.keyset(g["context"] - 1, g["w"], g["s"], lib=lib)) == g["held_tokens"]


# ---------------------------------------------------------------- backward

def _bwd_case(B=2, L=24, Hq=4, Hkv=2, d=16, seed=71):
    q, k, v = swa_inputs.prefill_inputs(B, L, Hq, Hkv, d, seed, sink_rows=2)
    g = torch.Generator("cpu").manual_seed(seed + 1)
    dout = torch.randn(B, L, Hq, d, generator=g, dtype=torch.float64)
    return q, k, v, dout


def check_backward_vs_sdpa_autograd(lib):
    """Gradients equal torch fp64 autograd through scaled_dot_product_attention
    with the same boolean mask (a library routine), GQA by repeated heads."""
    for (w, s) in ((6, 2), (24, 0), (1, 3)):
        q, k, v, dout = _bwd_case()
        B, L, Hq, d = q.shape
        G = Hq // k.shape[2]
        scale = 1.0 / math.sqrt(d)
        qd, kd, vd = (x.double().requires_grad_(True) for x in (q, k, v))
        mask = torch.from_numpy(oracle.swa_mask(L, w, s) & np.tril(np.ones((L, L), dtype=bool)))
        o = F.scaled_dot_product_attention(
            qd.permute(0, 2, 1, 3), kd.repeat_interleave(G, dim=2).permute(0, 2, 1, 3),
            vd.repeat_interleave(G, dim=2).permute(0, 2, 1, 3), attn_mask=mask,
            scale=float(np.float32(scale)))
        (o.permute(0, 2, 1, 3) * dout).sum().backward()
        dq, dk, dv = oracle.prefill_backward(q, k, v, dout, w, s, scale, lib=lib)
        for name, got, want in (("dq", dq, qd.grad), ("dk", dk, kd.grad), ("dv", dv, vd.grad)):
            want = want.numpy()
            err = np.abs(got - want).max() / max(np.abs(want).max(), 1e-300)
            assert err < 1e-10, (w, s, name, err)


def check_backward_window_one(lib):
    """w = 1, s = 0: out_t = v_t, so dv_t is the group's dout_t and dq = dk = 0."""
    q, k, v, dout = _bwd_case()
    Hkv = k.shape[2]
    dq, dk, dv = oracle.prefill_backward(q, k, v, dout, 1, 0, 0.25, lib=lib)
    assert not dq.any() and not dk.any()
    want = dout.numpy().reshape(dout.shape[0], dout.shape[1], Hkv, -1, dout.shape[3]).sum(3)
    assert np.allclose(dv, want, rtol=0, atol=1e-15)


def check_backward_key_shift_invariance(lib):
    """Adding one vector to every key leaves each softmax, hence every output,
    unchanged: the key gradients of a (b, KV head) sum to zero."""
    q, k, v, dout = _bwd_case()
    _, dk, _ = oracle.prefill_backward(q, k, v, dout, 7, 2, 0.25, lib=lib)
    tot = dk.sum(axis=1)                       # over positions -> [B, Hkv, d]
    assert np.abs(tot).max() <= 1e-12 * max(np.abs(dk).max(), 1.0)


def check_backward_euler_identity(lib):
    """Every output is linear in V: sum_j v_j . dv_j = sum_t dout_t . out_t."""
    q, k, v, dout = _bwd_case()
    _, _, dv = oracle.prefill_backward(q, k, v, dout, 5, 3, 0.25, lib=lib)
    out, _ = oracle.prefill(q, k, v, 5, 3, 0.25, lib=lib)
    lhs = float((v.double().numpy() * dv).sum())
    rhs = float((dout.numpy() * out).sum())
    assert abs(lhs - rhs) <= 1e-10 * max(abs(rhs), 1.0), (lhs, rhs)


ALL_CHECKS = [
    check_keymask_vs_pseudocode,
    check_counts_closed_form,
    check_full_window_is_causal,
    check_no_sinks_is_band,
    check_prefill_vs_sdpa,
    check_large_logits,
    check_full_causal_vs_sdpa_is_causal,
    check_window_one_identity,
    check_zero_query_mean,
    check_constant_values,
    check_gqa_equals_repeated_mha,
    check_weights_sum_to_one,
    check_weights_vs_torch_softmax,
    check_lse_vs_logsumexp,
    check_decode_equals_prefill_row,
    check_ring_page_example,
    check_ring_holds_keyset,
    check_footprint,
    check_backward_vs_sdpa_autograd,
    check_backward_window_one,
    check_backward_key_shift_invariance,
    check_backward_euler_identity,
]
