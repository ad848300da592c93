"""The fp64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin_fn", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin_fn):
    pin_fn(oracle.default())


def test_apply_is_shrink_then_expand():
    rng = np.random.default_rng(11)
    T, L, H1, H2, r = 9, 3, 16, 8, 4
    X = rng.standard_normal((T, H1))
    A = rng.standard_normal((L, H1, r))
    B = rng.standard_normal((L, r, H2))
    Y0 = rng.standard_normal((T, H2))
    perm = rng.permutation(T).astype(np.int32)
    seg_ptr, idx = [0, 3, 3, 8], [2, 0, -1]
    v = oracle.sgmv_shrink(X, A, seg_ptr, idx, perm)
    y1 = oracle.sgmv_expand(Y0, v, B, seg_ptr, idx, 0.25, perm)
    y2 = oracle.sgmv_apply(Y0, X, A, B, seg_ptr, idx, 0.25, perm)
    assert np.array_equal(y1, y2)


def test_widen_is_exact_for_half_types():
    import torch

    x = torch.randn(1000, generator=torch.Generator().manual_seed(0))
    for dt in (torch.float16, torch.bfloat16):
        h = x.to(dt)
        w = oracle.widen(h)
        assert w.dtype == np.float64
        assert torch.equal(torch.from_numpy(w).to(dt), h)


def test_oracle_rejects_bad_metadata():
    X = np.zeros((4, 8))
    A = np.zeros((2, 8, 2))
    with pytest.raises(ValueError):
        oracle.sgmv_shrink(X, A, [0, 5], [0])          # past T
    with pytest.raises(ValueError):
        oracle.sgmv_shrink(X, A, [0, 3, 2], [0, 1])    # decreasing
    with pytest.raises(ValueError):
        oracle.sgmv_shrink(X, A, [0, 2], [2])          # id == L
    with pytest.raises(ValueError):
        oracle.sgmv_shrink(X, A, [0, 2], [0], perm=[0, 4, 1, 2])
