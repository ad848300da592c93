"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Tolerance: max|dY| <= 1e-2 * RMS(Y_ref) (plus half an output ulp for bf16
outputs, see gpu_helpers.tolerance).  Segment metadata: bit-exact.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from rank_gemv_gb300 import workloads as wl
from tests.gpu_helpers import (assert_close, check_error_word, device_grouping, gpu_apply_rows,
                               oracle_apply_rows)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rank_gemv_gb300 import build, sgmv

    build.build()
    sgmv.load_library()
    sgmv.sgmv_get_device_error()  # start from a clear error word
    yield


def sg():
    from rank_gemv_gb300 import sgmv

    return sgmv


def _check_meta(perm, seg_ptr, idx, S, o_perm, o_seg, o_idx, T, L):
    s = int(S.item())
    assert s == len(o_idx)
    assert np.array_equal(perm.cpu().numpy()[:T], o_perm)
    sp = seg_ptr.cpu().numpy()
    ix = idx.cpu().numpy()
    assert np.array_equal(sp[: s + 1], o_seg)
    assert np.array_equal(ix[:s], o_idx)
    smax = sg().sgmv_max_segments(T, L)
    assert np.all(sp[s + 1: smax + 1] == T) and np.all(ix[s:smax] == -1)


# ---- the named workloads, in the benchmarked launch configuration ----------
@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("name", ["tiny", "decode-distinct", "decode-shared", "decode-zipf",
                                  "prefill"])
def test_workload_matches_oracle(name, seed):
    w = wl.make(name, seed, y0="randn" if seed else "zeros", shuffle_rows=bool(seed))
    y, perm, seg_ptr, idx, S = gpu_apply_rows(w)
    check_error_word(0)
    ref, o_perm, o_seg, o_idx = oracle_apply_rows(w)
    _check_meta(perm, seg_ptr, idx, S, o_perm, o_seg, o_idx, w.T, w.L)
    assert_close(y, ref, name)


def test_prefill_with_bf16_output():
    w = wl.make("prefill", 2, y_dtype=torch.bfloat16, y0="randn")
    y, *_ = gpu_apply_rows(w)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, "prefill bf16 Y")


def test_host_metadata_gives_the_same_bits():
    w = wl.make("decode-zipf", 4, y0="randn", shuffle_rows=True)
    y_dev, *_ = gpu_apply_rows(w)
    y_host, *_ = gpu_apply_rows(w, use_host_meta=True)
    check_error_word(0)
    assert torch.equal(y_dev, y_host)


# ---- shapes, ranks, dtypes ----------------------------------------------
def _mixed(T, L, H1, H2, r, dtype=torch.float16, y_dtype=None, seed=0):
    g = torch.Generator().manual_seed(seed)
    ra = torch.randint(-1, L, (T,), generator=g, dtype=torch.int32)
    return wl.draw(T, L, H1, H2, r, ra, dtype=dtype, y_dtype=y_dtype, y0="randn", seed=seed + 100,
                   scale=0.5)


@pytest.mark.parametrize("r", [1, 8, 15, 16, 17, 32, 48, 64, 100, 128])
def test_ranks(r):
    w = _mixed(37, 6, 264, 136, r, seed=r)
    y, *_ = gpu_apply_rows(w)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, f"r={r}")


@pytest.mark.parametrize("in_dt,y_dt", list(itertools.product(
    [torch.float16, torch.bfloat16], [torch.float16, torch.bfloat16, torch.float32])))
def test_dtypes(in_dt, y_dt):
    w = _mixed(29, 5, 1024, 520, 16, dtype=in_dt, y_dtype=y_dt, seed=3)
    y, *_ = gpu_apply_rows(w)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, f"{in_dt}->{y_dt}")


@pytest.mark.parametrize("H1,H2", [(8, 8), (24, 8), (8, 1032), (128, 136), (4104, 11016),
                                   (11008, 4096), (16384, 40)])
def test_ragged_and_small_dims(H1, H2):
    w = _mixed(19, 4, H1, H2, 16, seed=H1 + H2)
    y, *_ = gpu_apply_rows(w)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, f"H1={H1} H2={H2}")


def test_single_row_and_long_segment():
    w = wl.draw(1, 3, 512, 256, 16, [2], y0="randn")
    y, *_ = gpu_apply_rows(w)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, "T=1")
    w = wl.draw(45, 2, 512, 256, 16, [1] * 45, y0="randn", seed=5)
    y, *_ = gpu_apply_rows(w)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, "one segment of 45 rows")
    check_error_word(0)


# ---- explicit segment tables --------------------------------------------
def _explicit(seg_ptr, idx, T, L=4, H1=256, H2=136, r=8, perm=None, seed=7):
    g = torch.Generator().manual_seed(seed)
    w = wl.draw(T, L, H1, H2, r, torch.zeros(T, dtype=torch.int32), y0="randn", seed=seed,
                scale=1.25, generator=g)
    sp = torch.tensor(seg_ptr, dtype=torch.int32)
    ix = torch.tensor(idx, dtype=torch.int32)
    pm = None if perm is None else torch.tensor(perm, dtype=torch.int32)
    return w, sp, ix, pm


def _run_explicit(w, sp, ix, pm, host=False):
    y = w.Y0.to(DEV).clone()
    sg().sgmv_apply(y, w.X.to(DEV), w.A.to(DEV), w.B.to(DEV), sp.to(DEV), ix.to(DEV), w.scale,
                    perm=None if pm is None else pm.to(DEV), seg_ptr_host=sp if host else None)
    return y


@pytest.mark.parametrize("host", [False, True])
def test_empty_unsorted_shared_and_no_adapter_segments(host):
    # rows 0-1 uncovered; empty segment; adapter 3 before adapter 1; adjacent
    # segments sharing adapter 2; a no-adapter segment; rows 22-23 uncovered
    seg_ptr = [2, 2, 7, 9, 12, 20, 22]
    idx = [1, 3, 1, 2, 2, -1]
    T = 24
    perm = list(np.random.default_rng(0).permutation(T))
    w, sp, ix, pm = _explicit(seg_ptr, idx, T, perm=perm)
    y = _run_explicit(w, sp, ix, pm, host)
    check_error_word(0)
    ref = oracle.sgmv_apply(w.Y0, w.X, w.A, w.B, seg_ptr, idx, w.scale, perm=perm)
    assert_close(y, ref, "explicit segments")
    untouched = [perm[p] for p in (0, 1, 20, 21, 22, 23)]
    assert torch.equal(y[untouched].cpu(), w.Y0[untouched])


def test_invariants_hold_bitwise():
    T, L = 30, 4
    w, sp, ix, _ = _explicit([0, 12, 20, 30], [2, 0, 3], T, L=L)
    y = _run_explicit(w, sp, ix, None)
    # splitting a segment
    w2, sp2, ix2, _ = _explicit([0, 5, 12, 20, 23, 30], [2, 2, 0, 3, 3], T, L=L)
    assert torch.equal(y, _run_explicit(w2, sp2, ix2, None))
    # permuting segments permutes rows
    rows = list(range(20, 30)) + list(range(0, 12)) + list(range(12, 20))
    w3 = wl.Workload(**{**w.__dict__})
    w3.X, w3.Y0 = w.X[rows], w.Y0[rows]
    y3 = _run_explicit(w3, torch.tensor([0, 10, 22, 30], dtype=torch.int32),
                       torch.tensor([3, 2, 0], dtype=torch.int32), None)
    assert torch.equal(y3, y[rows])
    # B = 0 leaves Y unchanged
    w4 = wl.Workload(**{**w.__dict__})
    w4.B = torch.zeros_like(w.B)
    assert torch.equal(_run_explicit(w4, sp, ix, None).cpu(), w.Y0)
    # the same call twice gives the same bits
    assert torch.equal(y, _run_explicit(w, sp, ix, None))
    check_error_word(0)


# ---- shrink and expand as separate steps ---------------------------------
@pytest.mark.parametrize("r", [8, 16, 64, 128])
def test_shrink_and_expand_separately(r):
    w = _mixed(40, 5, 2048, 1032, r, seed=11 + r)
    perm, seg_ptr, idx, S = device_grouping(w.row_adapter, w.L)
    o_perm, o_seg, o_idx = oracle.build_segments(w.row_adapter, w.L)
    v = torch.full((w.T, r), float("nan"), device=DEV)
    sg().sgmv_shrink(v, w.X.to(DEV), w.A.to(DEV), seg_ptr, idx, perm=perm)
    check_error_word(0)
    v_ref = oracle.sgmv_shrink(w.X, w.A, o_seg, o_idx, perm=o_perm)
    assert_close(v, v_ref, "shrink v")
    # expand from a seeded v drawn by the input generator
    g = torch.Generator().manual_seed(5)
    v_in = torch.randn(w.T, r, generator=g)
    y = w.Y0.to(DEV).clone()
    sg().sgmv_expand(y, v_in.to(DEV), w.B.to(DEV), seg_ptr, idx, w.scale, perm=perm)
    check_error_word(0)
    ref = oracle.sgmv_expand(w.Y0, v_in, w.B, o_seg, o_idx, w.scale, perm=o_perm)
    assert_close(y, ref, "expand")
    # shrink then expand equals the oracle's whole update
    y2 = w.Y0.to(DEV).clone()
    sg().sgmv_expand(y2, v, w.B.to(DEV), seg_ptr, idx, w.scale, perm=perm)
    assert_close(y2, oracle.sgmv_apply(w.Y0, w.X, w.A, w.B, o_seg, o_idx, w.scale, perm=o_perm),
                 "shrink+expand")


@pytest.mark.parametrize("T,L,H1,r", [(128, 128, 4096, 16), (128, 2, 4096, 16), (128, 128, 11008, 16),
                                       (64, 128, 4096, 64)])
def test_shrink_at_decode_shapes(T, L, H1, r):
    """The standalone shrink at the Llama-2-7B projections' input widths, one
    row per adapter or a few shared adapters with rows of no adapter."""
    g = torch.Generator().manual_seed(T + L + H1 + r)
    ids = (torch.randperm(T, generator=g) % L).to(torch.int32) if L >= T else \
        torch.randint(-1, L, (T,), generator=g, dtype=torch.int32)
    w = wl.draw(T, L, H1, 64, r, ids, seed=H1 + r)
    perm, seg_ptr, idx, _ = device_grouping(w.row_adapter, w.L)
    o_perm, o_seg, o_idx = oracle.build_segments(w.row_adapter, w.L)
    v = torch.full((w.T, r), float("nan"), device=DEV)
    sg().sgmv_shrink(v, w.X.to(DEV), w.A.to(DEV), seg_ptr, idx, perm=perm)
    check_error_word(0)
    assert_close(v, oracle.sgmv_shrink(w.X, w.A, o_seg, o_idx, perm=o_perm), "shrink v")


# ---- device grouping ------------------------------------------------------
@pytest.mark.parametrize("T,L", [(1, 1), (8, 4), (32, 32), (64, 128), (100, 1), (2304, 8),
                                 (5000, 3000), (20000, 37), (777, 32767)])
def test_device_grouping_bit_exact(T, L):
    g = torch.Generator().manual_seed(T + L)
    ra = torch.randint(-1, L, (T,), generator=g, dtype=torch.int32)
    perm, seg_ptr, idx, S = device_grouping(ra, L)
    check_error_word(0)
    o_perm, o_seg, o_idx = oracle.build_segments(ra, L)
    _check_meta(perm, seg_ptr, idx, S, o_perm, o_seg, o_idx, T, L)


def test_device_grouping_reports_bad_id():
    ra = torch.tensor([0, 5, 1, -3, 1], dtype=torch.int32)
    perm, seg_ptr, idx, S = device_grouping(ra, 3)
    check_error_word(4)
    # bad ids are grouped as "no adapter"
    fixed = torch.tensor([0, -1, 1, -1, 1], dtype=torch.int32)
    o_perm, o_seg, o_idx = oracle.build_segments(fixed, 3)
    _check_meta(perm, seg_ptr, idx, S, o_perm, o_seg, o_idx, 5, 3)


# ---- errors reported by the kernels, never traps ---------------------------
def test_bad_adapter_index_is_skipped_and_reported():
    w, sp, ix, _ = _explicit([0, 4, 9, 12], [1, 7, 0], 12, L=4)
    y = _run_explicit(w, sp, ix, None)
    check_error_word(4)
    assert torch.equal(y[4:9].cpu(), w.Y0[4:9])
    # the other segments are applied as usual
    good = oracle.sgmv_apply(w.Y0, w.X, w.A, w.B, [0, 4, 9, 12], [1, -1, 0], w.scale)
    assert_close(y, good, "segments around the bad one")


def test_bad_segments_are_reported():
    w, sp, ix, _ = _explicit([0, 6, 3, 12], [1, 2, 0], 12, L=4)
    _run_explicit(w, sp, ix, None)
    check_error_word(8)
    w, sp, ix, _ = _explicit([0, 6, 40], [1, 2], 12, L=4)
    _run_explicit(w, sp, ix, None)
    check_error_word(8)


def test_bad_perm_entry_is_reported():
    w, sp, ix, pm = _explicit([0, 4, 8], [1, 2], 8, L=4, perm=[0, 1, 2, 3, 4, 5, 6, 99])
    y = _run_explicit(w, sp, ix, pm)
    check_error_word(4)
    ref = oracle.sgmv_apply(w.Y0, w.X, w.A, w.B, [0, 4, 7], [1, 2], w.scale,
                            perm=[0, 1, 2, 3, 4, 5, 6])
    assert_close(y[:7], ref[:7], "rows with valid perm entries")


def test_empty_problems():
    y = torch.zeros(0, 64, dtype=torch.float16, device=DEV)
    x = torch.zeros(0, 64, dtype=torch.float16, device=DEV)
    A = torch.zeros(2, 64, 8, dtype=torch.float16, device=DEV)
    B = torch.zeros(2, 8, 64, dtype=torch.float16, device=DEV)
    e = torch.zeros(1, dtype=torch.int32, device=DEV)
    sg().sgmv_apply(y, x, A, B, e, e[:0], 1.0)
    perm, seg_ptr, idx, S = device_grouping(torch.zeros(0, dtype=torch.int32), 3)
    assert int(S.item()) == 0 and int(seg_ptr[0].item()) == 0
    check_error_word(0)
