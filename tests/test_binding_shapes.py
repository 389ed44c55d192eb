"""The Python binding rejects tensors of the wrong shape before anything is
launched (CPU only: every case fails on its shapes, before the device checks).
The library takes the cache strides from w and s alone, so a cache built for
another (w, s), batch or head dimension must never reach a kernel."""
import pytest
import torch

import sliding_window_attention_05_b300 as swa

bf = torch.bfloat16


def _t(*shape, dtype=bf):
    return torch.zeros(*shape, dtype=dtype)


B, Hq, Hkv, d, w, s = 2, 8, 2, 64, 16, 4


@pytest.mark.parametrize("kc_shape", [
    (B, Hkv, s + w + 1, d),     # built for another window
    (B, Hkv, w, d),             # built without the sink slots
    (B + 1, Hkv, s + w, d),     # another batch
    (B, Hkv, s + w, 128),       # another head dimension
    (B, Hkv, (s + w) * d),      # not 4-D
])
def test_decode_rejects_cache_shape(kc_shape):
    q, pos = _t(B, Hq, d), torch.zeros(B, dtype=torch.int32)
    kc = _t(*kc_shape)
    with pytest.raises(ValueError, match="kcache"):
        swa.swa_decode(q, kc, kc.clone(), pos, w, s)
    with pytest.raises(ValueError, match="kcache"):
        swa.swa_append_decode(q, _t(B, Hkv, d), _t(B, Hkv, d), kc, kc.clone(), pos, w, s)
    with pytest.raises(ValueError, match="kcache"):
        swa.swa_prefill_chunk(_t(B, 5, Hq, d), _t(B, 5, Hkv, d), _t(B, 5, Hkv, d), kc,
                              kc.clone(), 0, w, s)


def test_decode_rejects_vcache_pos_and_out_shapes():
    q = _t(B, Hq, d)
    kc = _t(B, Hkv, s + w, d)
    pos = torch.zeros(B, dtype=torch.int32)
    with pytest.raises(ValueError, match="vcache"):
        swa.swa_decode(q, kc, _t(B, Hkv, s + w - 1, d), pos, w, s)
    with pytest.raises(ValueError, match="pos"):
        swa.swa_decode(q, kc, kc.clone(), torch.zeros(B + 1, dtype=torch.int32), w, s)
    with pytest.raises(ValueError, match="out"):
        swa.swa_decode(q, kc, kc.clone(), pos, w, s, out=_t(B, Hq, d + 8))
    with pytest.raises(ValueError, match="pos"):
        swa.swa_append_decode(q, _t(B, Hkv, d), _t(B, Hkv, d), kc, kc.clone(),
                              torch.zeros(1, dtype=torch.int32), w, s)
    with pytest.raises(ValueError, match="out"):
        swa.swa_append_decode(q, _t(B, Hkv, d), _t(B, Hkv, d), kc, kc.clone(), pos, w, s,
                              out=_t(B, Hq + 1, d))
    with pytest.raises(ValueError, match="k_new"):
        swa.swa_append_decode(q, _t(B, Hkv, d + 1), _t(B, Hkv, d + 1), kc, kc.clone(), pos, w, s)


def test_prefill_chunk_rejects_out_shape():
    kc = _t(B, Hkv, s + w, d)
    with pytest.raises(ValueError, match="out"):
        swa.swa_prefill_chunk(_t(B, 5, Hq, d), _t(B, 5, Hkv, d), _t(B, 5, Hkv, d), kc, kc.clone(),
                              0, w, s, out=_t(B, 6, Hq, d))


def test_prefill_rejects_out_shape():
    q, k = _t(1, 40, Hq, d), _t(1, 40, Hkv, d)
    with pytest.raises(ValueError, match="out"):
        swa.swa_prefill(q, k, k.clone(), w, s, out=_t(1, 39, Hq, d))
    with pytest.raises(ValueError, match="shape mismatch"):
        swa.swa_prefill(q, _t(1, 41, Hkv, d), _t(1, 41, Hkv, d), w, s)


def test_cache_append_rejects_shapes():
    kn = _t(B, 3, Hkv, d)
    kc = _t(B, Hkv, s + w, d)
    with pytest.raises(ValueError, match="cache"):
        swa.swa_cache_append(kn, kn.clone(), _t(B, Hkv, w, d), _t(B, Hkv, w, d),
                             torch.zeros(B, dtype=torch.int32), w, s)
    with pytest.raises(ValueError, match="pos_start"):
        swa.swa_cache_append(kn, kn.clone(), kc, kc.clone(), torch.zeros(B + 2, dtype=torch.int32),
                             w, s)
    with pytest.raises(ValueError, match="v_new"):
        swa.swa_cache_append(kn, _t(B, 4, Hkv, d), kc, kc.clone(),
                             torch.zeros(B, dtype=torch.int32), w, s)


def test_fa_decode_layer_needs_max_len():
    with pytest.raises(ValueError, match="max_len"):
        swa.AttentionLayer(1, 4, 1, 64, 16, 4, fa_decode=True)
    with pytest.raises(ValueError, match="max_len"):
        swa.HybridStack(1, 4, 1, 64, [(16, 4), (40, 0)], fa_decode=True)


def test_backward_rejects_shapes():
    L = 32
    q, k, v = _t(B, L, Hq, d), _t(B, L, Hkv, d), _t(B, L, Hkv, d)
    out, dout = _t(B, L, Hq, d), _t(B, L, Hq, d)
    lse = _t(B, Hq, L, dtype=torch.float32)
    with pytest.raises(ValueError):
        swa.swa_prefill_backward(q, k, _t(B, L, Hkv, 2 * d), out, dout, lse, w, s)
    with pytest.raises(ValueError):
        swa.swa_prefill_backward(q, k, v, _t(B, L + 1, Hq, d), dout, lse, w, s)
    with pytest.raises(ValueError):
        swa.swa_prefill_backward(q, k, v, out, _t(B, L, Hq + 1, d), lse, w, s)
    with pytest.raises(ValueError):
        swa.swa_prefill_backward(q, k, v, out, dout, _t(B, L, Hq, dtype=torch.float32), w, s)
    with pytest.raises(ValueError):
        swa.swa_prefill_backward(q, k, v, out, dout, lse, w, s, dk=_t(B, L, Hq, d))
