"""Chunked prefill into the ring cache on the GPU (through the C ABI): a
prompt prefilled chunk by chunk gives every row of the one-shot attention
(against the fp64 oracle) and leaves the cache bit-identical to appending the
whole prompt at once."""
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


CASES = [
    # B, L, Hq, Hkv, d, w, s, chunk lengths (summing to L)
    (1, 700, 8, 2, 64, 64, 4, [128, 128, 128, 128, 128, 60]),  # chunks past s + w - 1
    (2, 300, 32, 8, 128, 200, 4, [100, 100, 100]),            # chunks inside the first s + w - 1
    (1, 513, 4, 1, 128, 16, 0, [250, 1, 7, 255]),              # ragged, one-token chunk, no sinks
    (1, 400, 6, 2, 64, 50, 100, [30, 90, 280]),                # more sinks than window
    (1, 256, 4, 1, 64, 300, 4, [64, 64, 128]),                 # window longer than the prompt
    (3, 333, 12, 4, 64, 9, 2, [33, 100, 200]),                 # group of 3, tiny window
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_L%d_Hq%d_Hkv%d_d%d_w%d_s%d" % c[:7])
def test_chunked_prefill_equals_one_shot(case):
    B, L, Hq, Hkv, d, w, s, chunks = case
    assert sum(chunks) == L
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 7000 + L + w, sink_rows=min(s, 4))
    sc = scale_for(d)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    cache = swa.RingCache(B, Hkv, d, w, s, device=dev)
    outs, p = [], 0
    for T in chunks:
        outs.append(cache.prefill_chunk(qd[:, p:p + T].contiguous(), kd[:, p:p + T].contiguous(),
                                        vd[:, p:p + T].contiguous(), sc))
        p += T
    torch.cuda.synchronize()
    assert cache.length == L
    assert torch.equal(cache.next_pos.cpu(), torch.full((B,), L, dtype=torch.int32))
    ref, _ = oracle.prefill(q, k, v, w, s, sc)
    compare(torch.cat(outs, 1).cpu(), ref, f"chunked {chunks}")
    # the cache equals one append of the whole prompt
    whole = swa.RingCache(B, Hkv, d, w, s, device=dev)
    whole.append(kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(cache.k, whole.k) and torch.equal(cache.v, whole.v)


def test_chunked_prefill_then_decode():
    """Chunks, then token-by-token fused append + decode: every decoded row
    equals the oracle's row of the full sequence."""
    B, L, Hq, Hkv, d, w, s = 2, 260, 8, 2, 128, 40, 4
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 7100, sink_rows=4)
    sc = scale_for(d)
    dev = torch.device("cuda")
    cache = swa.RingCache(B, Hkv, d, w, s, device=dev)
    for a, b in ((0, 100), (100, 250)):
        cache.prefill_chunk(q[:, a:b].contiguous().to(dev), k[:, a:b].contiguous().to(dev),
                            v[:, a:b].contiguous().to(dev), sc)
    dec = [cache.step(q[:, t].to(dev), k[:, t].to(dev), v[:, t].to(dev), sc) for t in range(250, L)]
    torch.cuda.synchronize()
    rows = np.arange(250, L)
    ref, _ = oracle.prefill(q, k, v, w, s, sc, rows=rows)
    compare(torch.stack(dec, 1).cpu(), ref, "decode after chunks")


def test_long_chunked_prefill_sampled():
    """The SWA layer of the hybrid stack, SWA(2048, 100), B=1, L=16384,
    Hq=32, Hkv=8, d=128, in four chunks of 4096: sampled rows of every chunk."""
    B, L, Hq, Hkv, d, w, s, T = 1, 16384, 32, 8, 128, 2048, 100, 4096
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 7200)
    sc = scale_for(d)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    cache = swa.RingCache(B, Hkv, d, w, s, device=dev)
    outs = [cache.prefill_chunk(qd[:, p:p + T].contiguous(), kd[:, p:p + T].contiguous(),
                                vd[:, p:p + T].contiguous(), sc) for p in range(0, L, T)]
    torch.cuda.synchronize()
    out = torch.cat(outs, 1)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(4096 - 8, 4096 + 72),
                                     np.arange(L - 16, L), rng.integers(0, L, 48)]))
    ref, _ = oracle.prefill(q, k, v, w, s, sc, rows=rows)
    compare(out[:, torch.from_numpy(rows).to(dev)].cpu(), ref, "long chunked")


@pytest.mark.parametrize("P", [16, 64])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_L%d_Hq%d_Hkv%d_d%d_w%d_s%d" % c[:7])
def test_paged_chunked_prefill(case, P):
    """The same chunks over the paged layout: every row equals the oracle's,
    the pages a layer holds stay bounded, and decoding eight more tokens from
    the pages the chunks filled gives the oracle's rows."""
    B, L, Hq, Hkv, d, w, s, chunks = case
    extra = 8
    q, k, v = prefill_case(B, L + extra, Hq, Hkv, d, 7300 + L + w, sink_rows=min(s, 4))
    sc = scale_for(d)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    per_seq = -(-(L + extra) // P) + 2
    pool = swa.PagePool(B * per_seq, Hkv, d, page_size=P)
    cache = swa.PagedKVCache(pool, B, w, s, max_len=L + extra)
    outs, p = [], 0
    for T in chunks:
        outs.append(cache.prefill_chunk(qd[:, p:p + T].contiguous(), kd[:, p:p + T].contiguous(),
                                        vd[:, p:p + T].contiguous(), sc))
        p += T
        if w < L:
            bound = -(-s // P) + -(-(w - 1 + T) // P) + 1
            assert cache.pages_held() <= B * bound
    dec = []
    for t in range(L, L + extra):
        cache.append(kd[:, t:t + 1].contiguous(), vd[:, t:t + 1].contiguous())
        dec.append(cache.decode(qd[:, t].contiguous(), sc))
    torch.cuda.synchronize()
    ref, _ = oracle.prefill(q[:, :L], k[:, :L], v[:, :L], w, s, sc)
    compare(torch.cat(outs, 1).cpu(), ref, f"paged chunked {chunks}")
    ref, _ = oracle.prefill(q, k, v, w, s, sc, rows=np.arange(L, L + extra))
    compare(torch.stack(dec, 1).cpu(), ref, "paged decode after chunks")
    cache.release()
    assert pool.free_pages() == pool.n_pages


@pytest.mark.parametrize("mode", [swa.PREFILL_AUTO, swa.PREFILL_PAIR], ids=["auto", "pair"])
@pytest.mark.parametrize("paged", [False, True])
def test_chunk_writes_only_its_rows_of_out(paged, mode):
    """out is written in place by the prefill kernel, including the block
    that starts inside the staged prefix (copied with plain stores): the
    bytes around out stay untouched and every row is the oracle's. Both
    prefill kernels."""
    prev = swa.swa_prefill_select(mode)
    try:
        _chunk_rows_in_place(paged)
    finally:
        swa.swa_prefill_select(prev)


def _chunk_rows_in_place(paged):
    B, L, Hq, Hkv, d, w, s = 1, 420, 8, 2, 64, 200, 4   # Tq = 32 query positions per block
    q, k, v = prefill_case(B, L, Hq, Hkv, d, 7400, sink_rows=4)
    sc = scale_for(d)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    if paged:
        pool = swa.PagePool(64, Hkv, d, page_size=16)
        cache = swa.PagedKVCache(pool, B, w, s, max_len=L)
    else:
        cache = swa.RingCache(B, Hkv, d, w, s, device=dev)
    outs, p = [], 0
    # pos0 = 100 (prefix rows 0..99: 100 % 32 = 4) and pos0 = 250 (staged
    # prefix of s + w - 1 = 203 rows: 203 % 32 = 11), then 410 (also 203)
    for T in (100, 150, 160, 10):
        row = Hq * d
        guard = torch.full(((T + 64) * row,), 7.0, dtype=torch.bfloat16, device=dev)
        out = guard[32 * row:(32 + T) * row].view(1, T, Hq, d)
        cache.prefill_chunk(qd[:, p:p + T].contiguous(), kd[:, p:p + T].contiguous(),
                            vd[:, p:p + T].contiguous(), sc, out=out)
        torch.cuda.synchronize()
        assert (guard[:32 * row] == 7.0).all() and (guard[(32 + T) * row:] == 7.0).all(), T
        outs.append(out.clone())
        p += T
    ref, _ = oracle.prefill(q, k, v, w, s, sc)
    compare(torch.cat(outs, 1).cpu(), ref, "chunk rows in place")
