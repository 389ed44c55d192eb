"""The paged KV layout on the GPU (through the C ABI): paged append + paged
decode reproduce every prefill row (fp64 oracle), layers of both kinds share
one pool, and an unmapped page is reported through the device error word
without any copy being issued."""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_05_b300 as swa
from parity import compare, prefill_case, scale_for

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _device_error_clean():
    swa.swa_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert swa.swa_device_error(clear=True) == 0


@pytest.mark.parametrize("case", [
    # B, L, Hq, Hkv, d, w, s, page_size, prompt length
    (1, 256, 4, 1, 64, 64, 4, 16, 100),
    (2, 200, 32, 8, 128, 16, 4, 8, 1),
    (3, 150, 6, 2, 64, 9, 0, 4, 50),
    (1, 180, 8, 8, 128, 20, 30, 16, 60),
    (2, 130, 16, 2, 64, 200, 4, 32, 20),      # window beyond the sequence: a growing cache
    (1, 300, 32, 8, 128, 64, 4, 64, 128),
], ids=lambda c: "B%d_L%d_Hq%d_Hkv%d_d%d_w%d_s%d_P%d" % c[:8])
def test_paged_decode_equals_prefill_rows(case):
    """A prompt appended at once, then token-by-token paged append + decode:
    every decoded row equals the oracle's prefill row."""
    B, L, Hq, Hkv, d, w, s, P, L0 = case
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 8100 + L + P, sink_rows=min(s, 4))
    sc = scale_for(d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    pool = swa.PagePool(256, Hkv, d, page_size=P)
    cache = swa.PagedKVCache(pool, B, w, s, max_len=L)
    cache.append(kd[:, :L0].contiguous(), vd[:, :L0].contiguous())
    outs = [cache.decode(qd[:, L0 - 1].contiguous(), sc)]
    for t in range(L0, L):
        cache.append(kd[:, t:t + 1].contiguous(), vd[:, t:t + 1].contiguous())
        outs.append(cache.decode(qd[:, t].contiguous(), sc))
        if w < L:
            bound = -(-s // P) + -(-(w - 1) // P) + 1
            assert cache.pages_held() <= B * bound
    torch.cuda.synchronize()
    rows = np.arange(L0 - 1, L)
    ref, _ = oracle.prefill(q, k, v, w, s, sc, rows=rows)
    compare(torch.stack(outs, 1).cpu(), ref, "paged decode")
    cache.release()
    assert pool.free_pages() == 256


def test_hybrid_layers_share_one_pool():
    """An SWA(32, 4) layer and a full-attention layer draw pages from one pool
    while they step together; both decode correctly and the SWA layer's pages
    are recycled."""
    B, L, Hq, Hkv, d, P = 2, 240, 8, 2, 64, 16
    sc = scale_for(d)
    data = [prefill_case(B, L, Hq, Hkv, d, 8200 + i, sink_rows=4) for i in range(2)]
    pool = swa.PagePool(2 * B * (L // P + 2), Hkv, d, page_size=P)
    layers = [swa.PagedKVCache(pool, B, 32, 4, max_len=L), swa.PagedKVCache(pool, B, L, 0, max_len=L)]
    outs = [[], []]
    for t in range(L):
        for li, (layer, (q, k, v)) in enumerate(zip(layers, data)):
            layer.append(k[:, t:t + 1].contiguous().cuda(), v[:, t:t + 1].contiguous().cuda())
            outs[li].append(layer.decode(q[:, t].contiguous().cuda(), sc))
    torch.cuda.synchronize()
    assert layers[0].pages_held() <= B * (1 + 2 + 1)
    assert layers[1].pages_held() == B * (L // P)
    for li, ((q, k, v), (w, s)) in enumerate(zip(data, ((32, 4), (L, 0)))):
        ref, _ = oracle.prefill(q, k, v, w, s, sc)
        compare(torch.stack(outs[li], 1).cpu(), ref, f"layer {li}")


@pytest.mark.parametrize("bad", [-1, 1 << 20], ids=["unmapped", "out_of_range"])
def test_unmapped_page_is_reported(bad):
    """A table entry the decode needs is unmapped or names a page beyond the
    pool: the CTA issues no copy, writes nothing, and the device error word
    says so."""
    B, Hq, Hkv, d, w, s, P = 1, 4, 1, 64, 32, 4, 16
    _, k, v = prefill_case(B, 50, Hkv, Hkv, d, 8300)
    pool = swa.PagePool(16, Hkv, d, page_size=P)
    cache = swa.PagedKVCache(pool, B, w, s, max_len=64)
    cache.append(k.cuda(), v.cuda())
    q = torch.randn(B, Hq, d).to(torch.bfloat16).cuda()
    cache.table_dev[0, 2] = bad           # a window page of position 49
    out = torch.full_like(q, 7.0)
    cache.decode(q, out=out)
    torch.cuda.synchronize()
    assert swa.swa_device_error(clear=True) == 3
    assert bool((out == 7.0).all())        # nothing written
