"""The prefill kernel's tile schedule and in-tile mask, replayed on the GPU,
admit exactly the oracle's key sets (bit-exact, no pair twice)."""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_05_b300 as swa
from test_abi import SCHEDULE_CASES, _unpack

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=[swa.PREFILL_SINGLE, swa.PREFILL_PAIR], ids=["single", "pair"])
def kernel(request):
    """The device and host aids replay the tiling of the selected kernel."""
    prev = swa.swa_prefill_select(request.param)
    yield request.param
    swa.swa_prefill_select(prev)


@pytest.mark.parametrize("case", SCHEDULE_CASES, ids=lambda c: "L%d_Hq%d_Hkv%d_d%d_w%d_s%d" % c)
def test_device_keymask_matches_oracle(case):
    L, Hq, Hkv, d, w, s = case
    bits, counts = swa.swa_debug_keymask(L, Hq, Hkv, d, w, s, 0, L)
    torch.cuda.synchronize()
    want = oracle.keymask(L, w, s)
    assert np.array_equal(_unpack(bits.cpu(), L), want)
    assert np.array_equal(counts.cpu().numpy(), want.sum(axis=1))
    hb, hc = swa.swa_keymask_host(L, Hq, Hkv, d, w, s, 0, L)
    assert torch.equal(hb, bits.cpu()) and torch.equal(hc, counts.cpu())


@pytest.mark.parametrize("L,w,s", [(32768, 64, 4), (32768, 512, 4), (16384, 2048, 100)])
def test_device_keymask_large_rows(L, w, s):
    """Row windows of the long configurations, checked against the oracle."""
    for row0 in (0, w - 3, L // 2 - 17, L - 300):
        nrows = 300
        bits, counts = swa.swa_debug_keymask(L, 32, 8, 128, w, s, row0, nrows)
        torch.cuda.synchronize()
        got = _unpack(bits.cpu(), L)
        for r in range(0, nrows, 7):
            t = row0 + r
            want = np.zeros(L, dtype=bool)
            want[oracle.keyset(t, w, s)] = True
            assert np.array_equal(got[r], want), t
            assert counts[r].item() == want.sum()
