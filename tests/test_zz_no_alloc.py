"""sgmv_apply_noalloc: sgmv_apply for callers that may not allocate device memory.

Such callers (a plugin limited to its engine's pre-planned buffers, a serving
loop that forbids allocation after warm-up, code running under CUDA graph
capture) cannot hand sgmv_apply a workspace, so this entry point keeps the
tensor-core path's scratch in a fixed array inside the library.  The test runs
a prefill-shaped batch, whose long segments go through that scratch, twice in
a row through the C ABI and compares each result with sgmv_apply given a
workspace of its own and with the fp64 oracle, element by element, within the
parity tolerance of the other tests.  It also checks that a problem too large
for the fixed array is refused when it would need the array, and that a large
problem that can never reach the tensor cores (rank 16) runs without it and
matches the oracle.  This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
from rank_gemv_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, check_error_word, oracle_apply_rows

pytestmark = pytest.mark.gpu


def test_no_alloc_matches_apply_on_two_calls():
    from rank_gemv_gb300 import build, sgmv

    build.build()
    dev = torch.device("cuda")
    w = wl.make("prefill", 7, y0="randn", shuffle_rows=True)
    X, A, B = w.X.to(dev), w.A.to(dev), w.B.to(dev)
    perm, seg_ptr, idx, _ = sgmv.sgmv_build_segments_device(w.row_adapter.to(dev), w.L)
    ws = torch.empty(sgmv.sgmv_workspace_bytes(w.T, w.H1, w.H2, w.r), dtype=torch.uint8,
                     device=dev)
    y_ref = w.Y0.to(dev).clone()
    sgmv.sgmv_apply(y_ref, X, A, B, seg_ptr, idx, w.scale, perm=perm, workspace=ws)
    ref = y_ref.double().cpu().numpy()
    exact = oracle_apply_rows(w)[0]
    for _ in range(2):  # the second call finds the first call's contents in the scratch
        y = w.Y0.to(dev).clone()
        sgmv.sgmv_apply_noalloc(y, X, A, B, seg_ptr, idx, w.scale, perm=perm)
        assert sgmv.sgmv_last_launch_count() >= 2  # the tensor-core kernels ran
        check_error_word(0)
        assert_close(y, ref, "sgmv_apply_noalloc vs sgmv_apply")
        assert_close(y, exact, "sgmv_apply_noalloc vs oracle")


def test_no_alloc_refuses_problems_beyond_its_scratch():
    from rank_gemv_gb300 import sgmv

    dev = torch.device("cuda")
    T, H, r = 9000, 256, 128  # needs 9000 * 128 * 4 bytes > 4 MiB
    assert sgmv.sgmv_workspace_bytes(T, H, H, r) > 4 << 20
    x = torch.zeros(T, H, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(T, H, dtype=torch.float32, device=dev)
    A = torch.zeros(1, H, r, dtype=torch.bfloat16, device=dev)
    B = torch.zeros(1, r, H, dtype=torch.bfloat16, device=dev)
    seg_ptr = torch.tensor([0, T], dtype=torch.int32, device=dev)
    idx = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(sgmv.SgmvError) as e:
        sgmv.sgmv_apply_noalloc(y, x, A, B, seg_ptr, idx, 1.0)
    assert e.value.status == 6


def test_no_alloc_runs_large_low_rank_problems_without_scratch():
    """Rank 16 never reaches the tensor cores, so no scratch is needed however
    large the batch: a batch whose sgmv_workspace_bytes exceeds the fixed
    array still runs, on the CUDA cores, and matches the oracle."""
    from rank_gemv_gb300 import sgmv

    dev = torch.device("cuda")
    T, L, H, r = 66000, 3, 64, 16
    assert sgmv.sgmv_workspace_bytes(T, H, H, r) > 4 << 20
    g = torch.Generator().manual_seed(11)
    ids = torch.randint(-1, L, (T,), generator=g, dtype=torch.int32)
    w = wl.draw(T, L, H, H, r, ids, seed=11, y0="randn")
    perm, seg_ptr, idx = (t.to(dev) for t in sgmv.sgmv_build_segments(w.row_adapter, L))
    sph = sgmv.sgmv_build_segments(w.row_adapter, L)[1]
    y = w.Y0.to(dev).clone()
    sgmv.sgmv_apply_noalloc(y, w.X.to(dev), w.A.to(dev), w.B.to(dev), seg_ptr, idx, w.scale,
                            perm=perm, seg_ptr_host=sph)
    check_error_word(0)
    o_perm, o_seg, o_idx = oracle.build_segments(w.row_adapter, L)
    ref = oracle.sgmv_apply(w.Y0, w.X, w.A, w.B, o_seg, o_idx, w.scale, perm=o_perm)
    assert np.array_equal(sph.numpy(), o_seg)
    assert_close(y, ref, "large rank-16 batch through sgmv_apply_noalloc")
