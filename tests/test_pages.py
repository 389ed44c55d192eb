"""The host page allocator of the paged KV layout (CPU): after every
reservation a sequence maps exactly the logical pages that hold a position of
K(p) (checked against the key set enumerated from its definition), pages are
never shared, and the pool's count of free pages stays exact."""
import ctypes

import numpy as np
import pytest

import sliding_window_attention_05_b300 as swa

lib = swa.lib()


def key_pages(p: int, w: int, s: int, P: int) -> set:
    """Logical pages of the positions j <= p with j >= p - w + 1 or j < s."""
    return {j // P for j in range(p + 1) if j >= p - w + 1 or j < s}


class Pool:
    def __init__(self, n):
        self.h = ctypes.c_void_p(lib.swa_page_pool_create(n))
        assert self.h.value
        self.n = n

    def free(self):
        return lib.swa_page_pool_free_pages(self.h)

    def reserve(self, table, p, w, s, P):
        return lib.swa_paged_reserve(self.h, table.ctypes.data_as(ctypes.c_void_p), table.size,
                                     p, w, s, P)

    def release(self, table):
        return lib.swa_paged_release(self.h, table.ctypes.data_as(ctypes.c_void_p), table.size)

    def __del__(self):
        lib.swa_page_pool_destroy(self.h)


def mapped(table):
    return {int(i) for i in np.nonzero(table >= 0)[0]}


@pytest.mark.parametrize("w,s,P", [(100, 4, 16), (64, 0, 64), (7, 20, 8), (1, 1, 1), (50, 3, 128)])
def test_swa_layer_maps_exactly_its_key_pages(w, s, P):
    pool = Pool(400)
    table = np.full(1200 // P + 2, -1, dtype=np.int32)
    for p in list(range(0, 400)) + list(range(900, 1000, 7)):  # steps, then jumps
        assert pool.reserve(table, p, w, s, P) == swa.SWA_OK, swa.swa_last_error()
        assert mapped(table) == key_pages(p, w, s, P), p
        phys = table[table >= 0]
        assert len(set(phys.tolist())) == len(phys)          # no page mapped twice
        assert pool.free() == pool.n - len(phys)
    # a sliding-window layer's footprint stays bounded
    assert len(mapped(table)) <= -(-s // P) + -(-(w - 1) // P) + 1
    assert pool.release(table) == swa.SWA_OK
    assert pool.free() == pool.n and (table == -1).all()


def test_full_layer_grows_and_two_layers_share_a_pool():
    P, n = 32, 300
    pool = Pool(n)
    full = np.full(200, -1, dtype=np.int32)
    swl = np.full(200, -1, dtype=np.int32)
    for p in range(0, 5000, 13):
        assert pool.reserve(full, p, 1 << 30, 0, P) == swa.SWA_OK
        assert pool.reserve(swl, p, 256, 100, P) == swa.SWA_OK
        assert mapped(full) == set(range(p // P + 1))
        assert mapped(swl) == key_pages(p, 256, 100, P)
        both = np.concatenate([full[full >= 0], swl[swl >= 0]])
        assert len(set(both.tolist())) == len(both)           # layers never share a page
        assert pool.free() == n - len(both)


def test_exhausted_pool_changes_nothing():
    pool = Pool(3)
    table = np.full(64, -1, dtype=np.int32)
    assert pool.reserve(table, 40, 1 << 20, 0, 16) == swa.SWA_OK     # pages 0, 1, 2
    before = table.copy()
    assert pool.reserve(table, 48, 1 << 20, 0, 16) == swa.SWA_ERR_UNSUPPORTED
    assert "exhausted" in swa.swa_last_error()
    assert (table == before).all() and pool.free() == 0
    # a sliding window frees pages as it moves, so the same pool goes on
    t2 = np.full(64, -1, dtype=np.int32)
    assert pool.release(table) == swa.SWA_OK
    for p in range(0, 1000):
        assert pool.reserve(t2, p, 20, 0, 16) == swa.SWA_OK


def test_bad_arguments():
    pool = Pool(8)
    table = np.full(4, -1, dtype=np.int32)
    assert pool.reserve(table, 4 * 16, 10, 0, 16) == swa.SWA_ERR_UNSUPPORTED   # beyond the table
    assert pool.reserve(table, -1, 10, 0, 16) == swa.SWA_ERR_INVALID_ARG
    assert pool.reserve(table, 5, 0, 0, 16) == swa.SWA_ERR_INVALID_ARG
    assert pool.reserve(table, 5, 10, 0, 0) == swa.SWA_ERR_INVALID_ARG
    forged = np.array([5, -1, -1, -1], dtype=np.int32)                       # not handed out
    assert pool.release(forged) == swa.SWA_ERR_INVALID_ARG
    assert lib.swa_page_pool_create(0) is None
    assert lib.swa_page_pool_free_pages(None) == -1


@pytest.mark.parametrize("w,s,P", [(100, 4, 16), (64, 0, 64), (7, 20, 8), (300, 2, 32)])
def test_range_reserve_maps_the_union_of_key_pages(w, s, P):
    """swa_paged_reserve_range(lo, hi) maps the pages of every K(p), lo <= p <=
    hi (what a prompt chunk at lo .. hi reads and writes), releases the rest,
    and with lo = hi is exactly swa_paged_reserve."""
    pool, pool1 = Pool(400), Pool(400)
    table = np.full(1200 // P + 2, -1, dtype=np.int32)
    single = table.copy()
    lo = 0
    for T in [1, 37, 200, 5, 64, 128, 1, 300]:
        hi = lo + T - 1
        rc = lib.swa_paged_reserve_range(pool.h, table.ctypes.data_as(ctypes.c_void_p), table.size,
                                         lo, hi, w, s, P)
        assert rc == swa.SWA_OK, swa.swa_last_error()
        want = set().union(*(key_pages(p, w, s, P) for p in range(lo, hi + 1)))
        assert mapped(table) == want, (lo, hi)
        phys = table[table >= 0]
        assert len(set(phys.tolist())) == len(phys)
        assert pool.free() == pool.n - len(phys)
        rc = lib.swa_paged_reserve_range(pool1.h, single.ctypes.data_as(ctypes.c_void_p),
                                         single.size, hi, hi, w, s, P)
        assert rc == swa.SWA_OK and mapped(single) == key_pages(hi, w, s, P)
        lo = hi + 1
    assert lib.swa_paged_reserve_range(pool.h, table.ctypes.data_as(ctypes.c_void_p), table.size,
                                       lo, lo - 1, w, s, P) == swa.SWA_ERR_INVALID_ARG
    assert pool.release(table) == swa.SWA_OK and pool1.release(single) == swa.SWA_OK
    assert pool.free() == pool.n and pool1.free() == pool1.n
