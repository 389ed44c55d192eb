"""The backward of the SWA(w, s) prefill on the GPU (through the C ABI)
against the fp64 oracle's gradients (the chain rule applied to the forward
definition; the oracle's backward is pinned to torch autograd, a closed form
and two invariants on the CPU).

Tolerance. The kernels round three quantities to bf16 on the way (the softmax
weights P before dV = P^T dO, dS before dQ = dS K and dK = dS^T Q, and the
forward output O that enters D = dO . O), each with a relative rounding error
of at most 2^-9, and the gradients themselves are rounded to bf16. Over a whole
gradient tensor that gives a relative L2 error of a few 1e-3; the bound below
is rel-L2 <= 1.5e-2 and max-abs <= 3e-2 * max |reference|, per tensor."""
import math

import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_05_b300 as swa
from parity import compare, prefill_case, scale_for

pytestmark = pytest.mark.gpu

BWD_REL_L2 = 1.5e-2
BWD_MAX_ABS_FRAC = 3e-2


@pytest.fixture(autouse=True)
def _device_error_clean():
    swa.swa_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert swa.swa_device_error(clear=True) == 0


def _dout(B, L, Hq, d, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randn(B, L, Hq, d, generator=g).to(torch.bfloat16)


def _check_grads(got, want, what):
    for name, g, r in zip(("dq", "dk", "dv"), got, want):
        scale = max(float(np.abs(r).max()), 1e-30)
        compare(g.cpu(), r, f"{what} {name}", max_abs=BWD_MAX_ABS_FRAC * scale, rel_l2=BWD_REL_L2)


def _run(B, L, Hq, Hkv, d, w, s, seed, sink_rows=0):
    q, k, v = prefill_case(B, L, Hq, Hkv, d, seed, sink_rows=sink_rows)
    dout = _dout(B, L, Hq, d, seed + 1)
    sc = scale_for(d)
    dev = torch.device("cuda")
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, dout))
    lse = torch.empty(B, Hq, L, dtype=torch.float32, device=dev)
    out = swa.swa_prefill(qd, kd, vd, w, s, sc, lse=lse)
    dq, dk, dv = swa.swa_prefill_backward(qd, kd, vd, out, gd, lse, w, s, sc)
    torch.cuda.synchronize()
    ref = oracle.prefill_backward(q, k, v, dout.double(), w, s, sc)
    return (dq, dk, dv), ref, lse, (q, k, v)


@pytest.mark.parametrize("mode", [swa.PREFILL_AUTO, swa.PREFILL_PAIR], ids=["auto", "pair"])
def test_forward_lse_matches_oracle(mode):
    prev = swa.swa_prefill_select(mode)
    try:
        _lse_case()
    finally:
        swa.swa_prefill_select(prev)


def _lse_case():
    B, L, Hq, Hkv, d, w, s = 2, 300, 8, 2, 128, 40, 4
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 8100, sink_rows=4)
    sc = scale_for(d)
    lse = torch.empty(B, Hq, L, dtype=torch.float32, device="cuda")
    out = swa.swa_prefill(q.cuda(), k.cuda(), v.cuda(), w, s, sc, lse=lse)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.prefill(q, k, v, w, s, sc)
    compare(out.cpu(), ref_out, "out with lse")
    err = np.abs(lse.cpu().double().numpy() - ref_lse.transpose(0, 2, 1))
    assert err.max() < 1e-3, err.max()


def test_tiny_config_all_gradients():
    """B=1, L=256, Hq=4, Hkv=1, d=64, SWA(64, 4): every element of dq, dk, dv."""
    got, ref, _, _ = _run(1, 256, 4, 1, 64, 64, 4, 8200)
    _check_grads(got, ref, "tiny")


def test_llama_shaped_config_all_gradients():
    """B=1, L=4096, Hq=32, Hkv=8, d=128, SWA(128, 4), sink keys x4."""
    got, ref, _, _ = _run(1, 4096, 32, 8, 128, 128, 4, 8300, sink_rows=4)
    _check_grads(got, ref, "llama-shaped")


BWD_CASES = [
    # B, L, Hq, Hkv, d, w, s
    (2, 300, 8, 8, 128, 17, 3),     # MHA, ragged tail
    (1, 200, 12, 4, 64, 33, 5),     # group of 3
    (1, 97, 4, 1, 64, 500, 4),      # w >= L: full causal
    (1, 400, 4, 1, 64, 50, 200),    # 200 sinks: two sink key tiles
    (2, 520, 16, 2, 128, 100, 0),   # group of 8, no sinks
    (1, 129, 4, 1, 128, 128, 16),   # window and sinks on tile edges
    (1, 700, 32, 8, 128, 512, 4),   # long window, several tiles per block
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "B%d_L%d_Hq%d_Hkv%d_d%d_w%d_s%d" % c)
def test_edge_cases(case):
    B, L, Hq, Hkv, d, w, s = case
    got, ref, _, _ = _run(B, L, Hq, Hkv, d, w, s, 8400 + L, sink_rows=min(s, 4))
    _check_grads(got, ref, str(case))


def test_window_one_closed_form():
    """SWA(1, 0): out_t = v_t, so dq = dk = 0 and dv is the group's sum of dout
    (the oracle gives exact zeros; on the GPU dS = dP - D is the difference of
    two fp32 dot products of the same bf16 values summed in different orders,
    so dq and dk are rounding noise only)."""
    B, L, Hq, Hkv, d = 1, 200, 8, 2, 64
    (dq, dk, dv), ref, _, _ = _run(B, L, Hq, Hkv, d, 1, 0, 8500)
    assert not ref[0].any() and not ref[1].any()
    assert float(dq.abs().max()) < 1e-3 and float(dk.abs().max()) < 1e-3
    want = torch.from_numpy(ref[2])
    g = torch.Generator("cpu").manual_seed(8501)
    dout = torch.randn(B, L, Hq, d, generator=g).to(torch.bfloat16).double()
    assert torch.allclose(want, dout.view(B, L, Hkv, Hq // Hkv, d).sum(3), atol=1e-12)
    compare(dv.cpu(), ref[2], "w=1 dv")


def test_long_window_sweep_config():
    """B=2, L=8192, Hq=32, Hkv=8, d=128, SWA(512, 4) with x4 sink keys: the
    long-prefill geometry at a quarter of its length, every gradient element."""
    got, ref, _, _ = _run(2, 8192, 32, 8, 128, 512, 4, 8600, sink_rows=4)
    _check_grads(got, ref, "L=8192 w=512")
