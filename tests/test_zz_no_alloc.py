"""sgmv_apply_noalloc: sgmv_apply for callers that may not allocate device memory.

Such callers (a plugin limited to its engine's pre-planned buffers, a serving
loop that forbids allocation after warm-up, code running under CUDA graph
capture) cannot hand sgmv_apply a workspace, so this entry point keeps the
tensor-core path's scratch in a fixed array inside the library.  The test runs
a prefill-shaped batch, whose long segments go through that scratch, twice in
a row through the C ABI and compares each result with sgmv_apply given a
workspace of its own, within the parity tolerance of the other tests.  It also
checks that a problem too large for the fixed array is refused.  This file is
named so that pytest collects it last.
"""
import pytest
import torch

from rank_gemv_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, check_error_word

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
    for _ in range(2):  # the second call finds the first call's contents in the scratch
        y = w.Y0.to(dev).clone()
        sgmv.sgmv_apply_noalloc(y, X, A, B, seg_ptr, idx, w.scale, perm=perm)
        assert sgmv.sgmv_last_launch_count() >= 2  # the tensor-core kernels ran
        check_error_word(0)
        assert_close(y, ref, "sgmv_apply_noalloc vs sgmv_apply")


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
