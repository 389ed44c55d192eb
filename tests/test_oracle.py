"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(lib, check):
    check(lib)


def test_raw_pseudocode_differs_only_in_early_rows():
    """The page's mask admits sink columns j < s even when j > t. The oracle
    clamps them to causal; the two masks differ only in rows t < s - 1."""
    import numpy as np
    for L in (6, 12):
        for w in (1, 3, 20):
            for s in (0, 1, 4, 9):
                raw = oracle.swa_mask(L, w, s)
                clamped = oracle.keymask(L, w, s)
                rows = np.nonzero((raw != clamped).any(axis=1))[0]
                assert all(t < s - 1 for t in rows), (L, w, s, rows)
