"""sgmv_apply_multi: several projections with the same rows and segments
(a layer's q / k / v, or gate / up) in one launch of the streaming kernel.

Each case checks the result against three (or four) separate sgmv_apply
calls bit for bit -- the cluster size, and with it every row's summation
order, is the same -- and against the oracle, and how many kernels the call
launched.
"""
import pytest
import torch

import oracle
from rank_gemv_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, check_error_word

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


def problems(P, T, L, H1, H2, r, ra, dtype, y_dtype, seed, shared_x=False):
    out = []
    for k in range(P):
        w = wl.draw(T, L, H1, H2, r, ra, dtype=dtype, y_dtype=y_dtype, y0="randn", seed=seed + k)
        if shared_x and out:
            w.X = out[0].X  # the same rows for every problem
        out.append(w)
    return out


def run_case(ws, host_meta=False, expect_launches=None):
    sgmv = sg()
    ra = ws[0].row_adapter
    L = ws[0].L
    if host_meta:
        perm, seg_ptr, idx = sgmv.sgmv_build_segments(ra, L)
        meta = dict(perm=perm.to(DEV), seg_ptr_host=seg_ptr)
        seg_d, idx_d, S = seg_ptr.to(DEV), idx.to(DEV), None
    else:
        perm, seg_d, idx_d, _ = sgmv.sgmv_build_segments_device(ra.to(DEV), L)
        meta = dict(perm=perm)
        S = sgmv.sgmv_max_segments(ws[0].T, L)
    xs = [w.X.to(DEV) for w in ws]
    As = [w.A.to(DEV) for w in ws]
    Bs = [w.B.to(DEV) for w in ws]
    ys = [w.Y0.to(DEV) for w in ws]
    sgmv.sgmv_apply_multi(ys, xs, As, Bs, seg_d, idx_d, 0.5, S=S, **meta)
    n = sgmv.load_library().sgmv_last_launch_count()
    check_error_word(0)
    if expect_launches is not None:
        assert n == expect_launches
    for k, w in enumerate(ws):
        y1 = w.Y0.to(DEV)
        sgmv.sgmv_apply(y1, xs[k], As[k], Bs[k], seg_d, idx_d, 0.5, S=S, **meta)
        assert torch.equal(ys[k], y1), f"problem {k}: not the bits of a separate call"
        o_perm, o_seg, o_idx = oracle.build_segments(w.row_adapter, w.L)
        ref = oracle.sgmv_apply(w.Y0, w.X, w.A, w.B, o_seg, o_idx, 0.5, perm=o_perm)
        assert_close(ys[k], ref, f"problem {k}")
    check_error_word(0)


def test_llama7b_qkv_one_launch():
    ra = wl.stack_row_adapter(128)
    ws = problems(3, 128, 128, 4096, 4096, 16, ra, torch.float16, torch.float16, 100)
    run_case(ws, expect_launches=1)


def test_one_problem_through_the_multi_entry():
    ra = wl.stack_row_adapter(128)
    ws = problems(1, 128, 128, 11008, 4096, 16, ra, torch.float16, torch.float16, 150)
    run_case(ws, expect_launches=1)


def test_llama7b_gate_up_one_launch():
    ra = wl.stack_row_adapter(128)
    ws = problems(2, 128, 128, 4096, 11008, 16, ra, torch.float16, torch.float16, 200)
    run_case(ws, expect_launches=1)


@pytest.mark.parametrize("dtype,y_dtype", [(torch.bfloat16, torch.float32),
                                           (torch.float16, torch.bfloat16)])
def test_four_problems_shared_rows_skewed_ids(dtype, y_dtype):
    g = torch.Generator().manual_seed(5)
    ra = wl.zipf_ids(g, 96, 40).to(torch.int32)
    ra[::7] = -1  # rows of no adapter
    ws = problems(4, 96, 40, 1024, 520, 32, ra, dtype, y_dtype, 300, shared_x=True)
    run_case(ws, host_meta=True, expect_launches=1)


def test_small_batch_falls_back_to_separate_calls():
    # 32 rows: clusters of four CTAs, one tile each, so three problems do not
    # fit one launch; the call makes three
    ra = torch.arange(32, dtype=torch.int32)
    ws = problems(3, 32, 32, 4096, 4096, 16, ra, torch.float16, torch.float16, 400)
    run_case(ws, expect_launches=3)


def test_rank_above_the_streaming_kernel():
    # r = 128: the CUDA-core fused kernel, one call per problem
    g = torch.Generator().manual_seed(6)
    ra = torch.randint(0, 6, (40,), generator=g, dtype=torch.int32)
    ws = problems(2, 40, 6, 256, 264, 128, ra, torch.float16, torch.float32, 500)
    run_case(ws, host_meta=True, expect_launches=2)


@pytest.mark.parametrize("r,y_dtype", [(12, torch.float32), (64, torch.bfloat16)])
def test_ranks_of_the_multi_problem_instantiation(r, y_dtype):
    # r = 12 runs the rank-16 instantiation with masked columns, r = 64 the
    # rank-64 one; 128 rows on 40 adapters (one-CTA clusters)
    g = torch.Generator().manual_seed(r)
    ra = torch.randint(0, 40, (128,), generator=g, dtype=torch.int32)
    ws = problems(2, 128, 40, 2048, 1032, r, ra, torch.bfloat16, y_dtype, 600 + r)
    run_case(ws, host_meta=True, expect_launches=1)
