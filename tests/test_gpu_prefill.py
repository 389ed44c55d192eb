"""SWA(w, s) prefill on the GPU (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_05_b300 as swa
from parity import compare, sample_rows, prefill_case, scale_for

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _device_error_clean():
    swa.swa_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert swa.swa_device_error(clear=True) == 0


@pytest.fixture(autouse=True, params=[swa.PREFILL_AUTO, swa.PREFILL_PAIR], ids=["auto", "pair"])
def kernel(request):
    """Every test of this module runs once with the library's kernel choice
    and once with the two-block (pair) kernel."""
    prev = swa.swa_prefill_select(request.param)
    yield request.param
    swa.swa_prefill_select(prev)


def _run(q, k, v, w, s, scale):
    dev = torch.device("cuda")
    out = swa.swa_prefill(q.to(dev), k.to(dev), v.to(dev), w, s, scale)
    torch.cuda.synchronize()
    return out


def test_tiny_config_all_rows():
    """B=1, L=256, Hq=4, Hkv=1, d=64, SWA(64, 4): every output element."""
    q, k, v = prefill_case(1, 256, 4, 1, 64, 1001)
    sc = scale_for(64)
    out = _run(q, k, v, 64, 4, sc)
    ref, _ = oracle.prefill(q, k, v, 64, 4, sc)
    compare(out.cpu(), ref, "tiny")


def test_llama_shaped_config_all_rows():
    """B=1, L=4096, Hq=32, Hkv=8, d=128, SWA(128, 4), sink keys x4."""
    q, k, v = prefill_case(1, 4096, 32, 8, 128, 1002, sink_rows=4)
    sc = scale_for(128)
    out = _run(q, k, v, 128, 4, sc)
    ref, _ = oracle.prefill(q, k, v, 128, 4, sc)
    compare(out.cpu(), ref, "llama-shaped")


EDGE_CASES = [
    # B, L, Hq, Hkv, d, w, s
    (1, 1, 4, 1, 64, 64, 4),        # a single token
    (2, 300, 8, 8, 128, 17, 3),     # MHA (128 positions per block), ragged tail
    (1, 200, 12, 4, 64, 33, 5),     # group of 3: 126 of 128 tile rows used
    (1, 97, 4, 1, 64, 500, 4),      # w >= L: full causal
    (1, 97, 4, 1, 128, 40, 300),    # s > L: every key is a sink
    (1, 400, 4, 1, 64, 50, 200),    # two sink tiles
    (2, 520, 16, 2, 128, 100, 0),   # group of 8, no sinks
    (1, 1000, 32, 8, 128, 2048, 0), # full causal, many band tiles
    (3, 333, 2, 1, 64, 7, 1),       # tiny window, one sink
    (1, 129, 4, 1, 128, 128, 16),   # window and sinks on tile boundaries
    (1, 1100, 32, 8, 128, 512, 4),  # sinks at the end of each block's last band tile
    (2, 700, 8, 2, 128, 460, 40),   # the same with a 48-key sink box, ragged tail
    (1, 800, 1, 1, 64, 400, 10),    # the same, MHA, d = 64
]


@pytest.mark.parametrize("case", EDGE_CASES, ids=lambda c: "B%d_L%d_Hq%d_Hkv%d_d%d_w%d_s%d" % c)
def test_edge_cases(case):
    B, L, Hq, Hkv, d, w, s = case
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 2000 + L, sink_rows=min(s, L))
    sc = scale_for(d)
    out = _run(q, k, v, w, s, sc)
    ref, _ = oracle.prefill(q, k, v, w, s, sc)
    compare(out.cpu(), ref, str(case))


def test_window_one_is_identity_bitexact():
    """SWA(1, 0): each query sees only itself, p = 1, so out == v exactly."""
    B, L, Hq, Hkv, d = 2, 300, 8, 2, 128
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 3001)
    out = _run(q, k, v, 1, 0, scale_for(d)).cpu()
    want = v.repeat_interleave(Hq // Hkv, dim=2)
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))


def test_output_guard_bands_untouched():
    B, L, Hq, Hkv, d = 1, 130, 4, 1, 64
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 3002)
    n = B * L * Hq * d
    pad = 4096
    buf = torch.full((n + 2 * pad,), -7.25, dtype=torch.bfloat16, device="cuda")
    out = buf[pad:pad + n].view(B, L, Hq, d)
    swa.swa_prefill(q.cuda(), k.cuda(), v.cuda(), 16, 4, scale_for(d), out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == -7.25) and torch.all(buf[pad + n:] == -7.25)
    ref, _ = oracle.prefill(q, k, v, 16, 4, scale_for(d))
    compare(out.cpu(), ref, "guarded")


@pytest.mark.parametrize("w", [64, 256, 512])
def test_long_prefill_window_sweep_sampled(w):
    """B=2, L=32768, Hq=32, Hkv=8, d=128, s=4, sink keys x4: sampled rows,
    every head and batch."""
    B, L, Hq, Hkv, d, s = 2, 32768, 32, 8, 128, 4
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 1004 + w, sink_rows=4)
    sc = scale_for(d)
    out = _run(q, k, v, w, s, sc)
    rows = sample_rows(L, w, s, 4096, seed=w)
    ref, _ = oracle.prefill(q, k, v, w, s, sc, rows=rows)
    compare(out[:, torch.from_numpy(rows).cuda()].cpu(), ref, f"long w={w}")


@pytest.mark.parametrize("w,s", [(2048, 100), (16384 + 256, 0)], ids=["swa2048_100", "full"])
def test_hybrid_layer_prefill_sampled(w, s):
    """B=1, L=16384, Hq=32, Hkv=8, d=128: one SWA(2048, 100) layer and one full
    causal layer of the hybrid stack; sampled rows."""
    B, L, Hq, Hkv, d = 1, 16384, 32, 8, 128
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 1500 + s)
    sc = scale_for(d)
    out = _run(q, k, v, w, s, sc)
    # SWA layer: every row t < w + s + 128 = 2276; full layer: the first 4096
    # rows (each reaches position 0); both: the last 128 and 4096 random rows
    rows = sample_rows(L, w, s, 4096, seed=7, head_cap=4096)
    ref, _ = oracle.prefill(q, k, v, w, s, sc, rows=rows)
    compare(out[:, torch.from_numpy(rows).cuda()].cpu(), ref, f"hybrid w={w} s={s}")


def test_repeated_calls_are_deterministic():
    q, k, v = prefill_case(1, 1024, 32, 8, 128, 3003, sink_rows=4)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    a = swa.swa_prefill(qd, kd, vd, 256, 4)
    b = swa.swa_prefill(qd, kd, vd, 256, 4)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_host_buffers_path():
    """CPU tensors in, CPU tensor out (the end-to-end call)."""
    q, k, v = prefill_case(1, 512, 32, 8, 128, 3004, sink_rows=4)
    out = swa.swa_prefill(q, k, v, 128, 4)
    assert out.device.type == "cpu"
    ref, _ = oracle.prefill(q, k, v, 128, 4, scale_for(128))
    compare(out, ref, "host buffers")
