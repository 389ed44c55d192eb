"""The C ABI without a GPU: symbols, argument checks and the host-side index
logic (ring slots, cache sizing, the prefill tile schedule) against the oracle."""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import oracle_pins
import sliding_window_attention_05_b300 as swa

LIB = swa.lib()
NULL = None
P = ctypes.c_void_p(4096)  # a non-null, 16-byte aligned dummy (never dereferenced)


def test_header_symbols_are_exported():
    names = swa.header_functions()
    assert {"swa_prefill", "swa_cache_append", "swa_decode", "swa_decode_workspace_size",
            "swa_cache_slot", "swa_debug_keymask"} <= set(names)
    raw = ctypes.CDLL(swa.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"libswa.so does not export {n}"


def test_library_has_no_driver_dependency():
    # the CUDA runtime is static and the driver is looked up at run time, so the
    # library loads on a machine without a GPU driver
    out = os.popen(f"ldd {swa.LIB_PATH}").read()
    assert "libcuda.so" not in out and "libcudart.so" not in out, out


def test_status_strings():
    assert swa.swa_status_string(0) == "ok"
    assert "invalid" in swa.swa_status_string(1)
    assert "unsupported" in swa.swa_status_string(2)


def _prefill(q=P, k=P, v=P, o=P, B=1, L=16, Hq=4, Hkv=1, d=64, w=4, s=1, scale=0.125):
    return LIB.swa_prefill(q, k, v, o, B, L, Hq, Hkv, d, w, s, ctypes.c_float(scale), None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(q=NULL), 1), (dict(o=NULL), 1), (dict(k=ctypes.c_void_p(4100)), 1),
    (dict(B=0), 1), (dict(L=0), 1), (dict(w=0), 1), (dict(w=-3), 1), (dict(s=-1), 1),
    (dict(Hq=6, Hkv=4), 1), (dict(Hkv=0), 1), (dict(scale=0.0), 1), (dict(scale=-1.0), 1),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(d=96), 2), (dict(d=256), 2), (dict(Hq=256, Hkv=1), 2),
])
def test_prefill_rejects_bad_arguments(kwargs, status):
    assert _prefill(**kwargs) == status
    assert swa.swa_last_error()


def test_append_and_decode_reject_bad_arguments():
    ap = LIB.swa_cache_append
    assert ap(P, P, P, P, NULL, 1, 1, 1, 64, 4, 1, None) == 1
    assert ap(P, P, P, P, P, 1, 0, 1, 64, 4, 1, None) == 1
    assert ap(P, P, P, P, P, 1, 1, 1, 64, 0, 1, None) == 1
    assert ap(P, P, P, P, P, 1, 1, 1, 80, 4, 1, None) == 2
    dec = LIB.swa_decode
    f = ctypes.c_float(0.1)
    assert dec(P, P, P, NULL, P, 1, 4, 1, 64, 4, 1, f, NULL, 0, None) == 1
    assert dec(P, P, P, P, P, 1, 4, 3, 64, 4, 1, f, NULL, 0, None) == 1
    assert dec(P, P, P, P, P, 1, 4, 1, 64, 4, 1, ctypes.c_float(0.0), NULL, 0, None) == 1
    # a long cache with few sequences needs split-KV workspace
    need = swa.swa_decode_workspace_size(1, 32, 8, 128, 16640, 0)
    assert need > 0
    assert dec(P, P, P, P, P, 1, 32, 8, 128, 16640, 0, f, NULL, 0, None) == 1
    assert dec(P, P, P, P, P, 1, 32, 8, 128, 16640, 0, f, P, need - 1, None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_returns_error():
    assert _prefill() in (3, 4)


def test_decode_workspace_sizes():
    # 64 sequences x 8 KV heads fill the GPU without splitting the cache
    assert swa.swa_decode_workspace_size(64, 32, 8, 128, 64, 4) == 0
    # one sequence over a 2148-slot cache is split
    assert swa.swa_decode_workspace_size(1, 32, 8, 128, 2048, 100) > 0
    assert swa.swa_decode_workspace_size(1, 32, 8, 128, 0, 4) == 0


def test_decode_split_policy_invariants():
    # The split count is visible through the workspace: B * Hq * splits rows of
    # d fp32 partial outputs plus one (max, sum) pair. Whatever the shape, every
    # split must fit what one decode CTA stages at once (256 slots), no split
    # may be thinner than the 64-slot floor the policy keeps, and an unsplit
    # cache must itself fit one CTA.
    for B in (1, 2, 3, 8, 16, 64, 256):
        for Hkv, G in ((1, 1), (2, 3), (8, 4), (8, 8), (4, 32)):
            Hq = Hkv * G
            for w, s in ((1, 0), (64, 4), (252, 4), (300, 4), (512, 4), (2048, 100),
                         (16640, 0), (262144, 0)):
                cap = s + w
                for d in (64, 128):
                    ws = swa.swa_decode_workspace_size(B, Hq, Hkv, d, w, s)
                    if ws == 0:
                        assert cap <= 256, (B, Hq, Hkv, d, w, s)
                        continue
                    row = B * Hq * (4 * d + 8)
                    assert ws % row == 0, (B, Hq, Hkv, d, w, s, ws)
                    splits = ws // row
                    assert 2 <= splits <= -(-cap // 64), (B, Hq, Hkv, d, w, s, splits)
                    assert -(-cap // splits) <= 256, (B, Hq, Hkv, d, w, s, splits)


def test_cache_slot_matches_ring_simulation():
    for w in (1, 2, 3, 4, 7, 64, 100):
        for s in (0, 1, 4, 5, 100):
            for last in list(range(0, 3 * (s + w) + 5)) + [4095, 65536, 262143]:
                slots = oracle.ring_contents(last, w, s)
                for i, p in enumerate(slots.tolist()):
                    if p >= 0:
                        assert swa.swa_cache_slot(p, w, s) == i, (w, s, last, p)
    assert swa.swa_cache_slot(-1, 4, 0) == -1
    assert swa.swa_cache_slot(3, 0, 0) == -1


def test_cache_slot_page_example():
    g = oracle_pins.golden()["ring_eviction"]
    held = {swa.swa_cache_slot(p, g["w"], g["s"]): p for p in range(g["tokens_appended"])}
    # the 5th token (position 4) took the slot of the 1st (position 0)
    assert held[swa.swa_cache_slot(0, g["w"], g["s"])] == 4
    assert sorted(held.values()) == g["held_positions"]


def test_cache_bytes_page_examples():
    g = oracle_pins.golden()["kv_cache_bytes"]
    # the cache holds every token when the window spans the whole input
    per_layer = 2 * swa.swa_cache_bytes(1, g["n_kv"], g["d_q"], g["seq"], 0)  # K and V
    total = g["layers"] * per_layer
    assert total == 2 * g["layers"] * g["seq"] * g["d_q"] * g["n_kv"] * g["bytes_per_value"]
    assert abs(total - g["approx_bytes"]) / g["approx_bytes"] < g["rel_tol"]
    g = oracle_pins.golden()["kv_saving_long_context"]
    full = swa.swa_cache_bytes(1, 8, 128, g["seq"], 0)
    win = swa.swa_cache_bytes(1, 8, 128, g["w"], 0)
    assert 1.0 - win / full == g["saving"]
    g = oracle_pins.golden()["sink_window_footprint"]
    assert swa.swa_cache_bytes(1, 1, 128, g["w"], g["s"]) == g["held_tokens"] * 128 * 2


@pytest.fixture(params=[swa.PREFILL_SINGLE, swa.PREFILL_PAIR], ids=["single", "pair"])
def prefill_mode(request):
    """Runs a test once per prefill kernel (the plan and key-mask aids follow it)."""
    prev = swa.swa_prefill_select(request.param)
    yield request.param
    swa.swa_prefill_select(prev)


def test_prefill_select_rejects_unknown_modes():
    assert LIB.swa_prefill_select(3) == -1 and LIB.swa_prefill_select(-1) == -1
    with pytest.raises(ValueError):
        swa.swa_prefill_select(7)


def test_prefill_plan(prefill_mode):
    p = swa.swa_prefill_plan(4096, 32, 8, 128, 128, 4)
    assert p["Tq"] == 32 and p["rows"] == 128
    assert p["n_band"] % 16 == 0 and p["n_band"] <= 192
    assert p["s_box"] == 16 and p["n_sink"] == 1
    assert p["stages"] >= 2
    if prefill_mode == swa.PREFILL_SINGLE:
        # the whole steady-state span (w + Tq - 1 = 159 keys) fits one band tile
        assert p["n_band"] >= 128 + 31
    else:
        # a pair's span (w + 2 Tq - 1 = 191 keys) in two tiles of at most 128
        # keys, the sink box riding in the first: 16 + 112 = 128 columns
        assert p["n_band"] == 112 and 2 * p["n_band"] >= 191
        assert p["stages"] >= 4
    p = swa.swa_prefill_plan(300, 12, 4, 64, 40, 200)
    assert p["Tq"] == 42 and p["rows"] == 126
    assert p["n_sink"] == 2 and p["s_box"] == 112


def _unpack(bits: torch.Tensor, L: int) -> np.ndarray:
    b = bits.numpy().view(np.uint32)
    out = np.zeros((b.shape[0], L), dtype=bool)
    for j in range(L):
        out[:, j] = (b[:, j // 32] >> np.uint32(j % 32)) & 1
    return out


SCHEDULE_CASES = [
    # L, Hq, Hkv, d, w, s
    (256, 4, 1, 64, 64, 4),
    (300, 32, 8, 128, 128, 4),
    (300, 8, 8, 128, 17, 3),
    (200, 12, 4, 64, 33, 5),
    (150, 8, 1, 128, 1, 0),
    (150, 4, 2, 64, 16, 0),
    (97, 4, 1, 64, 500, 4),
    (97, 4, 1, 128, 40, 300),
    (400, 4, 1, 64, 50, 200),
    (640, 32, 8, 128, 512, 100),
    (1, 4, 1, 64, 64, 4),
    # the sink box rides at the end of a block's last band tile (three 192-key
    # band tiles whose last one owns at most 192 - s_box keys)
    (1100, 32, 8, 128, 512, 4),
    (1500, 32, 8, 64, 470, 16),
    (800, 1, 1, 64, 400, 10),
    (700, 8, 2, 128, 460, 40),
]


@pytest.mark.parametrize("case", SCHEDULE_CASES, ids=lambda c: "L%d_Hq%d_Hkv%d_d%d_w%d_s%d" % c)
def test_host_schedule_matches_oracle_keysets(case, prefill_mode):
    L, Hq, Hkv, d, w, s = case
    bits, counts = swa.swa_keymask_host(L, Hq, Hkv, d, w, s, 0, L)
    got = _unpack(bits, L)
    want = oracle.keymask(L, w, s)
    assert np.array_equal(got, want)
    # no key admitted twice (sink and band tiles are disjoint)
    assert np.array_equal(counts.numpy(), want.sum(axis=1))


def test_host_schedule_exhaustive_small(prefill_mode):
    for L in (1, 5, 31, 32, 33, 70):
        for (Hq, Hkv) in ((1, 1), (4, 1), (6, 2), (8, 1)):
            for w in (1, 2, 3, 16, 17, 33, 64, 100):
                for s in (0, 1, 4, 16, 17, 40):
                    bits, counts = swa.swa_keymask_host(L, Hq, Hkv, 64, w, s, 0, L)
                    want = oracle.keymask(L, w, s)
                    assert np.array_equal(_unpack(bits, L), want), (L, Hq, Hkv, w, s)
                    assert np.array_equal(counts.numpy(), want.sum(axis=1)), (L, Hq, Hkv, w, s)


def test_schedule_skips_out_of_window_tiles(prefill_mode):
    """Keys multiplied per query block stay O(w + Tq + sink tile), not O(t)."""
    L, Hq, Hkv, d, w, s = 32768, 32, 8, 128, 512, 4
    p = swa.swa_prefill_plan(L, Hq, Hkv, d, w, s)
    bits, counts = swa.swa_keymask_host(L, Hq, Hkv, d, w, s, L - 64, 64)
    assert counts.numpy().max() == w + s
    blocks = 1 if prefill_mode == swa.PREFILL_SINGLE else 2   # query blocks per item
    visited = p["n_band"] * -(-(w + blocks * p["Tq"] - 1) // p["n_band"]) + p["s_box"]
    assert visited < 2 * (w + s)


def test_hybrid_layer_windows():
    """Even layers SWA(2048, 100); odd layers full causal, written as a window
    that covers the prompt and every decode step, with no sinks."""
    win = swa.hybrid_layer_windows(8, 16384, 256)
    assert win[0::2] == [(2048, 100)] * 4
    assert win[1::2] == [(16640, 0)] * 4
    # a full-causal window never evicts: every position the run reaches keeps its slot
    w, s = win[1]
    slots = [swa.swa_cache_slot(p, w, s) for p in range(0, 16384 + 256, 97)]
    assert slots == list(range(0, 16384 + 256, 97))


def test_prefill_chunk_rejects_bad_arguments():
    lib = swa.lib()
    dummy = ctypes.c_void_p(4096)
    args = dict(B=1, T=64, Hq=8, Hkv=2, d=64, w=32, s=4, pos0=100)

    def call(ws=dummy, nbytes=1 << 30, **kw):
        a = dict(args, **kw)
        return lib.swa_prefill_chunk(dummy, dummy, dummy, dummy, dummy, dummy, a["B"], a["T"],
                                     a["Hq"], a["Hkv"], a["d"], a["w"], a["s"], a["pos0"],
                                     ctypes.c_float(0.125), ws, nbytes, None)

    assert call(pos0=-1) == swa.SWA_ERR_INVALID_ARG
    assert call(T=0) == swa.SWA_ERR_INVALID_ARG
    assert call(w=0) == swa.SWA_ERR_INVALID_ARG
    assert call(Hq=7) == swa.SWA_ERR_INVALID_ARG
    assert call(d=96) == swa.SWA_ERR_UNSUPPORTED
    need = swa.swa_prefill_chunk_workspace_size(1, 64, 8, 2, 64, 32, 4, 100)
    assert call(nbytes=need - 1) == swa.SWA_ERR_INVALID_ARG
    assert "workspace" in swa.swa_last_error()
    assert call(ws=None) == swa.SWA_ERR_INVALID_ARG


def test_prefill_chunk_workspace_size():
    """k and v over min(pos0, s + w - 1) + T staged rows (q and out are not
    staged), plus the append's positions: it stops growing once pos0 passes
    s + w - 1, and does not depend on Hq."""
    f = swa.swa_prefill_chunk_workspace_size
    assert f(1, 64, 8, 2, 64, 32, 4, -1) == 0
    assert f(1, 64, 8, 2, 64, 0, 4, 0) == 0
    row = (2 * 2) * 64 * 2                  # bytes of one staged row of k, v
    assert f(1, 64, 8, 2, 64, 32, 4, 35) == f(1, 64, 32, 2, 64, 32, 4, 35)
    a, b = f(1, 64, 8, 2, 64, 32, 4, 0), f(1, 64, 8, 2, 64, 32, 4, 35)
    assert b - a == 35 * row
    assert f(1, 64, 8, 2, 64, 32, 4, 10_000) == f(1, 64, 8, 2, 64, 32, 4, 35)
    assert a >= 64 * row


def test_backward_and_lse_reject_bad_arguments():
    """The prefill with lse and the backward check their arguments before any
    device call (no GPU needed)."""
    f = ctypes.c_float(0.125)
    bwd = LIB.swa_prefill_backward
    ws_need = swa.swa_prefill_backward_workspace_size(1, 64, 8, 2, 64, 4)
    assert ws_need > 0

    def call(lse=P, ws=P, nbytes=ws_need, B=1, L=64, Hq=8, Hkv=2, d=64, w=16, s=4, scale=f, q=P):
        return bwd(q, P, P, P, P, lse, P, P, P, B, L, Hq, Hkv, d, w, s, scale, ws, nbytes, None)

    assert call(q=NULL) == swa.SWA_ERR_INVALID_ARG
    assert call(lse=NULL) == swa.SWA_ERR_INVALID_ARG
    assert call(lse=ctypes.c_void_p(4098)) == swa.SWA_ERR_INVALID_ARG   # lse not 4-byte aligned
    assert call(L=0) == swa.SWA_ERR_INVALID_ARG
    assert call(w=0) == swa.SWA_ERR_INVALID_ARG
    assert call(Hq=6, Hkv=4) == swa.SWA_ERR_INVALID_ARG
    assert call(scale=ctypes.c_float(0.0)) == swa.SWA_ERR_INVALID_ARG
    assert call(d=96) == swa.SWA_ERR_UNSUPPORTED
    assert call(nbytes=ws_need - 1) == swa.SWA_ERR_INVALID_ARG
    assert "workspace" in swa.swa_last_error()
    lse = LIB.swa_prefill_lse
    assert lse(P, P, P, P, NULL, 1, 64, 8, 2, 64, 16, 4, f, None) == swa.SWA_ERR_INVALID_ARG
    assert lse(P, P, P, P, ctypes.c_void_p(4097), 1, 64, 8, 2, 64, 16, 4, f,
               None) == swa.SWA_ERR_INVALID_ARG
    assert lse(NULL, P, P, P, P, 1, 64, 8, 2, 64, 16, 4, f, None) == swa.SWA_ERR_INVALID_ARG
    assert lse(P, P, P, P, P, 1, 64, 8, 2, 80, 16, 4, f, None) == swa.SWA_ERR_UNSUPPORTED


def test_paged_prefill_chunk_rejects_bad_arguments():
    f = ctypes.c_float(0.125)
    fn = LIB.swa_paged_prefill_chunk
    need = swa.swa_prefill_chunk_workspace_size(1, 64, 8, 2, 64, 32, 4, 100)

    def call(table=P, P_=16, max_pages=64, n_pages=32, T=64, pos0=100, ws=P, nbytes=need, d=64):
        return fn(P, P, P, P, P, table, P, 1, T, 8, 2, d, P_, max_pages, n_pages, 32, 4, pos0, f,
                  ws, nbytes, None)

    assert call(table=NULL) == swa.SWA_ERR_INVALID_ARG
    assert call(P_=0) == swa.SWA_ERR_INVALID_ARG
    assert call(max_pages=0) == swa.SWA_ERR_INVALID_ARG
    assert call(n_pages=0) == swa.SWA_ERR_INVALID_ARG
    assert call(T=0) == swa.SWA_ERR_INVALID_ARG
    assert call(pos0=-1) == swa.SWA_ERR_INVALID_ARG
    assert call(d=96) == swa.SWA_ERR_UNSUPPORTED
    assert call(nbytes=need - 1) == swa.SWA_ERR_INVALID_ARG
