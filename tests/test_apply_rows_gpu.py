"""sgmv_apply_rows (grouping + update in one call) against the oracle.

Up to 64 rows it is one kernel in which every CTA groups the batch itself;
otherwise it is the grouping kernel followed by sgmv_apply.  Both must give the oracle's result and its metadata bit-exact,
and the single-kernel form must give the same bits as the two-call form.
"""
import numpy as np
import pytest
import torch

import oracle
from rank_gemv_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, check_error_word, oracle_apply_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def sg():
    from rank_gemv_gb300 import sgmv

    return sgmv


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rank_gemv_gb300 import build

    build.build()
    sg().load_library()
    sg().sgmv_get_device_error()
    yield


def meta_buffers(T, L):
    smax = sg().sgmv_max_segments(T, L)
    return (torch.full((max(T, 1),), -7, dtype=torch.int32, device=DEV),
            torch.full((smax + 1,), -7, dtype=torch.int32, device=DEV),
            torch.full((max(smax, 1),), -7, dtype=torch.int32, device=DEV),
            torch.full((1,), -7, dtype=torch.int32, device=DEV))


def run_rows(w, with_meta=True, ws=False):
    y = w.Y0.to(DEV).clone()
    out = meta_buffers(w.T, w.L) if with_meta else None
    work = None
    if ws:
        work = torch.empty(sg().sgmv_workspace_bytes(w.T, w.H1, w.H2, w.r), dtype=torch.uint8,
                           device=DEV)
    sg().sgmv_apply_rows(y, w.X.to(DEV), w.A.to(DEV), w.B.to(DEV), w.row_adapter.to(DEV),
                         w.scale, out=out, workspace=work)
    return y, out, sg().sgmv_last_launch_count()


def check_meta(out, w):
    perm, seg_ptr, idx, S = (t.cpu().numpy() for t in out)
    o_perm, o_seg, o_idx = oracle.build_segments(w.row_adapter, w.L)
    s = int(S[0])
    assert s == len(o_idx)
    assert np.array_equal(perm[: w.T], o_perm)
    assert np.array_equal(seg_ptr[: s + 1], o_seg)
    assert np.array_equal(idx[:s], o_idx)
    smax = sg().sgmv_max_segments(w.T, w.L)
    assert np.all(seg_ptr[s + 1: smax + 1] == w.T) and np.all(idx[s:smax] == -1)


@pytest.mark.parametrize("shuffle", [False, True])
@pytest.mark.parametrize("name", ["tiny", "decode-distinct", "decode-shared", "decode-zipf"])
def test_decode_workloads(name, shuffle):
    w = wl.make(name, 3, y0="randn", shuffle_rows=shuffle)
    y, out, launches = run_rows(w)
    assert launches == (1 if w.T <= 64 else 2)
    check_error_word(0)
    check_meta(out, w)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, name)
    if w.T <= 64:
        y2, _, _ = run_rows(w, with_meta=False)
        assert torch.equal(y, y2)


@pytest.mark.parametrize("T", [33, 47, 64])
@pytest.mark.parametrize("r", [16, 36, 64])
def test_grouped_batches_above_32_rows(T, r):
    """One-launch batches above 32 rows are cut into two-row tiles: skewed ids
    (some rows without an adapter), odd T and ranks that are not a multiple
    of 16 must give the oracle's result, and the two-call form's bits."""
    g = torch.Generator().manual_seed(100 * T + r)
    L = 40
    ra = wl.zipf_ids(g, T, L)
    ra[torch.randperm(T, generator=g)[:3]] = -1
    w = wl.draw(T, L, 1024, 1032, r, ra, dtype=torch.float16, y0="randn", seed=T + r)
    y_one, out, launches = run_rows(w)
    assert launches == 1
    check_error_word(0)
    check_meta(out, w)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y_one, ref, f"T={T} r={r}")
    y_two = w.Y0.to(DEV).clone()
    perm, seg_ptr, idx, _ = sg().sgmv_build_segments_device(w.row_adapter.to(DEV), w.L)
    sg().sgmv_apply(y_two, w.X.to(DEV), w.A.to(DEV), w.B.to(DEV), seg_ptr, idx, w.scale,
                    perm=perm)
    check_error_word(0)
    assert torch.equal(y_one, y_two)


def test_same_bits_as_grouping_then_apply():
    w = wl.make("decode-zipf", 8, y0="randn", shuffle_rows=True)
    y_one, *_ = run_rows(w)
    y_two = w.Y0.to(DEV).clone()
    perm, seg_ptr, idx, _ = sg().sgmv_build_segments_device(w.row_adapter.to(DEV), w.L)
    sg().sgmv_apply(y_two, w.X.to(DEV), w.A.to(DEV), w.B.to(DEV), seg_ptr, idx, w.scale,
                    perm=perm)
    check_error_word(0)
    assert torch.equal(y_one, y_two)


@pytest.mark.parametrize("T,expect_launches", [(1, 1), (63, 1), (64, 1), (65, 2), (600, 2)])
def test_batch_size_boundary(T, expect_launches):
    g = torch.Generator().manual_seed(T)
    ra = torch.randint(-1, 40, (T,), generator=g, dtype=torch.int32)  # adapters 40..47 unused
    w = wl.draw(T, 48, 512, 264, 16, ra, y0="randn", seed=T, scale=0.5)
    y, out, launches = run_rows(w)
    assert launches == expect_launches
    check_error_word(0)
    check_meta(out, w)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, f"T={T}")


def test_prefill_with_tensor_cores():
    w = wl.make("prefill", 4, y0="randn", shuffle_rows=True)
    y, out, launches = run_rows(w, ws=True)
    assert launches >= 3  # grouping, then (CUDA-core) + tensor-core shrink + expand
    check_error_word(0)
    check_meta(out, w)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, "prefill")


def test_bad_ids_are_no_adapter_and_reported():
    ra = torch.tensor([0, 9, 1, -5, 1, 2], dtype=torch.int32)
    w = wl.draw(6, 3, 256, 128, 8, ra, y0="randn", seed=2)
    y, out, _ = run_rows(w)
    check_error_word(4)
    fixed = torch.tensor([0, -1, 1, -1, 1, 2], dtype=torch.int32)
    w_fixed = wl.Workload(**{**w.__dict__})
    w_fixed.row_adapter = fixed
    ref, *_ = oracle_apply_rows(w_fixed)
    assert_close(y, ref, "bad ids")
    check_meta(out, w_fixed)


def test_large_batch_needs_metadata_buffers():
    w = wl.draw(100, 4, 256, 128, 8, torch.zeros(100, dtype=torch.int32))
    with pytest.raises(sg().SgmvError) as e:
        run_rows(w, with_meta=False)
    assert e.value.status == 1
