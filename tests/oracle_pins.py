"""Pins for the fp64 oracle: checks that tie it to something other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` if the
oracle disagrees with what the pages or plain mathematics fix:
  - hand-worked fixtures under ``tests/golden/`` (values computed by hand);
  - special cases that reduce to a library routine (numpy matmul, numpy's
    stable argsort);
  - the check the pages themselves suggest: a batch mixing adapters must
    equal each adapter's model run alone on its own rows ("Punica: when LoRA
    fine-tuned models need multi-tenant serving", omica.com.cn article, §5.2,
    troubleshooting row on output quality);
  - closed forms (selector adapters, one-hot rows, zero B, zero scale);
  - invariants: splitting a segment, permuting segments, no-adapter rows;
  - brute-force enumeration of every small grouping problem.
``test_oracle_pins.py`` runs them on the real oracle; ``test_oracle_mutants.py``
runs them on broken copies of it and expects each copy to fail at least one.
"""
from __future__ import annotations

import itertools

import numpy as np

from tests.golden import load

ALL_PINS = []


def pin(fn):
    ALL_PINS.append(fn)
    return fn


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_problem(rng, T, L, H1, H2, r):
    X = rng.standard_normal((T, H1))
    A = rng.standard_normal((L, H1, r)) / np.sqrt(H1)
    B = rng.standard_normal((L, r, H2)) / np.sqrt(r)
    Y0 = rng.standard_normal((T, H2))
    return X, A, B, Y0


def _group_with_numpy(row_adapter):
    """Segments from numpy's stable argsort (a library routine)."""
    ra = np.asarray(row_adapter)
    perm = np.argsort(ra, kind="stable").astype(np.int32)
    ids, counts = np.unique(ra, return_counts=True)
    seg_ptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return perm, seg_ptr, ids.astype(np.int32)


# -- hand-worked fixtures -----------------------------------------------------
@pin
def pin_worked_example(o):
    d = load("sgmv_worked_example.txt")
    v = o.sgmv_shrink(d["X"], d["A"], d["seg_ptr"], d["idx"])
    assert np.array_equal(v, d["v"]), (v, d["v"])
    Y = o.sgmv_apply(d["Y0"], d["X"], d["A"], d["B"], d["seg_ptr"], d["idx"], d["scale"])
    assert np.array_equal(Y, d["Y"]), (Y, d["Y"])
    Y2 = o.sgmv_expand(d["Y0"], d["v"], d["B"], d["seg_ptr"], d["idx"], d["scale"])
    assert np.array_equal(Y2, d["Y"])


@pin
def pin_worked_example_permuted_rows(o):
    """The fixture with its rows stored in another physical order."""
    d = load("sgmv_worked_example.txt")
    T = d["T"]
    pi = np.array([3, 5, 0, 4, 1, 2], np.int32)  # physical row of sorted position p
    Xp = np.zeros_like(d["X"])
    Y0p = np.zeros_like(d["Y0"])
    Xp[pi] = d["X"]
    Y0p[pi] = d["Y0"]
    Y = o.sgmv_apply(Y0p, Xp, d["A"], d["B"], d["seg_ptr"], d["idx"], d["scale"], perm=pi)
    for p in range(T):
        assert np.array_equal(Y[pi[p]], d["Y"][p])


@pin
def pin_worked_grouping(o):
    d = load("segments_worked_example.txt")
    perm, seg_ptr, idx = o.build_segments(d["row_adapter"], d["L"])
    assert np.array_equal(perm, d["perm"])
    assert np.array_equal(seg_ptr, d["seg_ptr"])
    assert np.array_equal(idx, d["idx"])


# -- special cases that reduce to library routines ----------------------------
@pin
def pin_single_adapter_is_dense_product(o):
    """All rows on one adapter: SGMV is the dense X @ A[a] @ B[a]."""
    rng = _rng(1)
    T, L, H1, H2, r, a, scale = 7, 3, 24, 20, 5, 2, 0.75
    X, A, B, Y0 = _rand_problem(rng, T, L, H1, H2, r)
    seg_ptr, idx = np.array([0, T], np.int32), np.array([a], np.int32)
    v = o.sgmv_shrink(X, A, seg_ptr, idx)
    assert np.allclose(v, X @ A[a], rtol=1e-12, atol=1e-12)
    Y = o.sgmv_apply(Y0, X, A, B, seg_ptr, idx, scale)
    assert np.allclose(Y, Y0 + scale * (X @ A[a]) @ B[a], rtol=1e-12, atol=1e-12)


@pin
def pin_mixed_batch_equals_each_adapter_alone(o):
    """A batch that mixes adapters (rows stored unsorted, some rows without an
    adapter, some adapters unused) equals each adapter applied alone, as a
    dense product, to its own rows."""
    rng = _rng(2)
    T, L, H1, H2, r, scale = 23, 5, 16, 12, 3, -1.25
    X, A, B, Y0 = _rand_problem(rng, T, L, H1, H2, r)
    ra = rng.integers(-1, L - 1, size=T).astype(np.int32)  # adapter L-1 unused
    perm, seg_ptr, idx = _group_with_numpy(ra)
    Y = o.sgmv_apply(Y0, X, A, B, seg_ptr, idx, scale, perm=perm)
    ref = Y0.copy()
    for a in range(L):
        rows = np.nonzero(ra == a)[0]
        if rows.size:
            ref[rows] = Y0[rows] + scale * (X[rows] @ A[a]) @ B[a]
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
    v = o.sgmv_shrink(X, A, seg_ptr, idx, perm=perm)
    for p in range(T):
        t = perm[p]
        want = X[t] @ A[ra[t]] if ra[t] >= 0 else np.zeros(r)
        assert np.allclose(v[p], want, rtol=1e-12, atol=1e-12)


# -- closed forms -------------------------------------------------------------
@pin
def pin_selector_adapters(o):
    """A[a] = [I_r; 0] and B[a] = [I_r | 0]: the delta is X's first r columns."""
    rng = _rng(3)
    T, L, H1, H2, r, scale = 5, 2, 6, 5, 4, 0.5
    X, A, B, Y0 = _rand_problem(rng, T, L, H1, H2, r)
    A[1] = 0.0
    A[1, :r, :r] = np.eye(r)
    B[1] = 0.0
    B[1, :r, :r] = np.eye(r)
    seg_ptr, idx = np.array([0, T], np.int32), np.array([1], np.int32)
    v = o.sgmv_shrink(X, A, seg_ptr, idx)
    assert np.array_equal(v, X[:, :r])
    Y = o.sgmv_apply(Y0, X, A, B, seg_ptr, idx, scale)
    want = Y0.copy()
    want[:, :r] += scale * X[:, :r]
    assert np.array_equal(Y, want)


@pin
def pin_one_hot_row_picks_a_row_of_A(o):
    rng = _rng(4)
    T, L, H1, H2, r = 4, 3, 9, 7, 6
    X, A, B, Y0 = _rand_problem(rng, T, L, H1, H2, r)
    X[:] = 0.0
    hs = [0, 3, 8, 5]
    for t, h in enumerate(hs):
        X[t, h] = 1.0
    seg_ptr, idx = np.array([0, 2, 4], np.int32), np.array([2, 1], np.int32)
    v = o.sgmv_shrink(X, A, seg_ptr, idx)
    for t, h in enumerate(hs):
        assert np.array_equal(v[t], A[idx[t // 2], h])


@pin
def pin_zero_B_or_zero_scale_keeps_Y(o):
    rng = _rng(5)
    T, L, H1, H2, r = 9, 3, 8, 10, 4
    X, A, B, Y0 = _rand_problem(rng, T, L, H1, H2, r)
    seg_ptr, idx = np.array([0, 4, 9], np.int32), np.array([0, 2], np.int32)
    Bz = np.zeros_like(B)
    assert np.array_equal(o.sgmv_apply(Y0, X, A, Bz, seg_ptr, idx, 1.0), Y0)
    assert np.array_equal(o.sgmv_apply(Y0, X, A, B, seg_ptr, idx, 0.0), Y0)


@pin
def pin_delta_scales_with_scale(o):
    """With Y0 = 0 the result is scale times the delta (exact for powers of two)."""
    rng = _rng(6)
    T, L, H1, H2, r = 6, 2, 8, 8, 3
    X, A, B, _ = _rand_problem(rng, T, L, H1, H2, r)
    Y0 = np.zeros((T, H2))
    seg_ptr, idx = np.array([0, 3, 6], np.int32), np.array([1, 0], np.int32)
    y1 = o.sgmv_apply(Y0, X, A, B, seg_ptr, idx, 1.0)
    y4 = o.sgmv_apply(Y0, X, A, B, seg_ptr, idx, 4.0)
    assert np.array_equal(y4, 4.0 * y1)
    assert np.abs(y1).max() > 0


# -- invariants ---------------------------------------------------------------
@pin
def pin_splitting_a_segment_changes_nothing(o):
    rng = _rng(7)
    T, L, H1, H2, r = 10, 4, 12, 9, 3
    X, A, B, Y0 = _rand_problem(rng, T, L, H1, H2, r)
    y = o.sgmv_apply(Y0, X, A, B, [0, 6, 10], [3, 1], 1.5)
    y_split = o.sgmv_apply(Y0, X, A, B, [0, 2, 6, 10], [3, 3, 1], 1.5)
    assert np.array_equal(y, y_split)
    v = o.sgmv_shrink(X, A, [0, 6, 10], [3, 1])
    v_split = o.sgmv_shrink(X, A, [0, 2, 2, 6, 10], [3, 0, 3, 1])  # plus an empty segment
    assert np.array_equal(v, v_split)


@pin
def pin_permuting_segments_permutes_rows(o):
    rng = _rng(8)
    L, H1, H2, r = 4, 10, 7, 2
    lens = [3, 1, 4]
    ids = [2, 0, 3]
    T = sum(lens)
    X, A, B, Y0 = _rand_problem(rng, T, L, H1, H2, r)
    seg_ptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    y = o.sgmv_apply(Y0, X, A, B, seg_ptr, ids, 0.5)
    order = [2, 0, 1]
    rows = np.concatenate([np.arange(seg_ptr[s], seg_ptr[s + 1]) for s in order])
    lens2 = [lens[s] for s in order]
    seg_ptr2 = np.concatenate([[0], np.cumsum(lens2)]).astype(np.int32)
    y2 = o.sgmv_apply(Y0[rows], X[rows], A, B, seg_ptr2, [ids[s] for s in order], 0.5)
    assert np.array_equal(y2, y[rows])


@pin
def pin_rows_without_adapter_are_untouched(o):
    rng = _rng(9)
    T, L, H1, H2, r = 12, 3, 8, 8, 2
    X, A, B, Y0 = _rand_problem(rng, T, L, H1, H2, r)
    # rows 0-1 before the first segment, rows 10-11 after the last one,
    # rows 4-6 in a segment without an adapter
    seg_ptr, idx = np.array([2, 4, 7, 10], np.int32), np.array([1, -1, 2], np.int32)
    y = o.sgmv_apply(Y0, X, A, B, seg_ptr, idx, 1.0)
    for t in [0, 1, 4, 5, 6, 10, 11]:
        assert np.array_equal(y[t], Y0[t])
    for t in [2, 3, 7, 8, 9]:
        assert not np.array_equal(y[t], Y0[t])
    v = o.sgmv_shrink(X, A, seg_ptr, idx)
    assert np.array_equal(v[4:7], np.zeros((3, r)))


# -- grouping -----------------------------------------------------------------
@pin
def pin_grouping_matches_stable_argsort_exhaustively(o):
    """Every row -> id assignment over ids {-1, 0, 1, 2} for T = 0..5."""
    L = 3
    for T in range(6):
        for ra in itertools.product(range(-1, L), repeat=T):
            ra = np.array(ra, np.int32)
            perm, seg_ptr, idx = o.build_segments(ra, L)
            if T == 0:
                assert perm.size == 0 and idx.size == 0 and list(seg_ptr) == [0]
                continue
            p2, s2, i2 = _group_with_numpy(ra)
            assert np.array_equal(perm, p2), (ra, perm, p2)
            assert np.array_equal(seg_ptr, s2), (ra, seg_ptr, s2)
            assert np.array_equal(idx, i2), (ra, idx, i2)


@pin
def pin_grouping_invariants_large(o):
    rng = _rng(10)
    for T, L in [(1, 1), (64, 128), (1000, 37), (4096, 8)]:
        ra = rng.integers(-1, L, size=T).astype(np.int32)
        perm, seg_ptr, idx = o.build_segments(ra, L)
        S = idx.size
        assert seg_ptr[0] == 0 and seg_ptr[S] == T
        assert np.all(np.diff(seg_ptr) > 0)
        assert np.all(np.diff(idx) > 0)
        assert np.array_equal(np.sort(perm), np.arange(T))
        for s in range(S):
            rows = perm[seg_ptr[s]:seg_ptr[s + 1]]
            assert np.all(ra[rows] == idx[s])
            assert np.all(np.diff(rows) > 0)  # original order kept within an id
    try:
        o.build_segments(np.array([0, 3], np.int32), 3)
    except ValueError:
        pass
    else:
        raise AssertionError("id == L accepted")


# -- fused base linear + LoRA (y = xW + xAB) ------------------------------------
# "Punica: when LoRA fine-tuned models need multi-tenant serving", §2.1: the
# LoRA layer is y = xW + xAB = x(W + AB), so a row on adapter a must equal x
# times the merged weight W + scale * A[a] B[a] (numpy matmul), and a row of no
# adapter x W alone.


@pin
def pin_fused_rows_equal_the_merged_weight(o):
    rng = _rng(20)
    T, L, H1, H2, r, scale = 23, 4, 24, 40, 5, 0.75
    X, A, B, _ = _rand_problem(rng, T, L, H1, H2, r)
    W = rng.standard_normal((H1, H2)) / np.sqrt(H1)
    ra = rng.integers(-1, L, size=T).astype(np.int32)
    perm, seg_ptr, idx = _group_with_numpy(ra)
    Y = o.fused_linear_lora(X, W, A, B, seg_ptr, idx, scale, perm)
    for t in range(T):
        Wt = W if ra[t] < 0 else W + scale * (A[ra[t]] @ B[ra[t]])
        assert np.allclose(Y[t], X[t] @ Wt, rtol=1e-12, atol=1e-12), t


@pin
def pin_fused_without_adapters_is_the_base_product(o):
    rng = _rng(21)
    T, L, H1, H2, r = 9, 2, 17, 12, 3
    X, A, B, _ = _rand_problem(rng, T, L, H1, H2, r)
    W = rng.standard_normal((H1, H2))
    Y = o.fused_linear_lora(X, W, A, B, [0, T], [-1], 2.0)
    assert np.allclose(Y, X @ W, rtol=1e-12, atol=1e-12)
    # and rows outside every segment keep the base output too
    Y2 = o.fused_linear_lora(X, W, A, B, [0, 4], [1], 2.0)
    assert np.allclose(Y2[4:], X[4:] @ W, rtol=1e-12, atol=1e-12)
    assert np.allclose(Y2[:4], X[:4] @ (W + 2.0 * A[1] @ B[1]), rtol=1e-12, atol=1e-12)


@pin
def pin_fused_closed_form(o):
    # all-ones inputs: every base output is H1, every LoRA delta scale * H1 * r
    T, L, H1, H2, r, scale = 5, 3, 6, 7, 4, 0.5
    X, W = np.ones((T, H1)), np.ones((H1, H2))
    A, B = np.ones((L, H1, r)), np.ones((L, r, H2))
    Y = o.fused_linear_lora(X, W, A, B, [0, 2, 5], [2, -1], scale)
    assert np.array_equal(Y[:2], np.full((2, H2), H1 + scale * H1 * r))
    assert np.array_equal(Y[2:], np.full((3, H2), float(H1)))
