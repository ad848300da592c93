"""The latency-vs-batch micro-benchmark's methods agree.

bench.py --figure times the base layer alone, the base plus a per-adapter loop
of torch matmuls, and the base plus SGMV.  On small cases the loop and SGMV
must give the same y (up to the loop's own fp16 rounding of each adapter's
delta), and base + SGMV must match the fp64 oracle applied to the base output.
"""
import pytest
import torch

import bench
import oracle
from tests.gpu_helpers import assert_close, check_error_word

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.mark.parametrize("T,n", [(1, 1), (16, 4), (96, 96), (128, 7)])
def test_loop_and_sgmv_agree(T, n):
    from rank_gemv_gb300 import build, sgmv

    build.build()
    sgmv.load_library()
    g = torch.Generator().manual_seed(T + n)
    H1, H2, r, L = 512, 264, 16, 128
    W = (torch.randn(H1, H2, generator=g) * H1 ** -0.5).half().to(DEV)
    A = (torch.randn(L, H1, r, generator=g) * H1 ** -0.5).half().to(DEV)
    B = (torch.randn(L, r, H2, generator=g) * r ** -0.5).half().to(DEV)
    fns, err, (x, ids, y) = bench.figure_point(sgmv, DEV, W, A, B, T, n, seed=T)
    assert err < 2e-2, err
    fns["base"]()
    y0 = y.cpu().clone()
    fns["sgmv"]()
    check_error_word(0)
    perm, seg_ptr, idx = oracle.build_segments(ids, L)
    ref = oracle.sgmv_apply(y0, x.cpu(), A.cpu(), B.cpu(), seg_ptr, idx, 1.0, perm=perm)
    assert_close(y, ref, f"base + SGMV, T={T}, adapters={n}")
