"""Tensor-core (tcgen05) path for long segments against the fp64 oracle.

sgmv_apply sends segments to the tensor cores when it is given a workspace and
r is 64 or 128: all of them when segments average 8 rows or more, else those
of at least 64 rows, the shorter ones going to the CUDA-core kernel in the
same call.
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


def workspace(w):
    n = sg().sgmv_workspace_bytes(w.T, w.H1, w.H2, w.r)
    return torch.empty(n, dtype=torch.uint8, device=DEV)


def run(w, host_meta=False, ws=True):
    y = w.Y0.to(DEV).clone()
    X, A, B = w.X.to(DEV), w.A.to(DEV), w.B.to(DEV)
    if host_meta:
        perm, seg_ptr, idx = sg().sgmv_build_segments(w.row_adapter, w.L)
        sg().sgmv_apply(y, X, A, B, seg_ptr.to(DEV), idx.to(DEV), w.scale, perm=perm.to(DEV),
                        seg_ptr_host=seg_ptr, workspace=workspace(w) if ws else None)
    else:
        perm, seg_ptr, idx, _ = sg().sgmv_build_segments_device(w.row_adapter.to(DEV), w.L)
        sg().sgmv_apply(y, X, A, B, seg_ptr, idx, w.scale, perm=perm,
                        workspace=workspace(w) if ws else None)
    return y


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("y_dtype", [torch.float32, torch.bfloat16])
def test_prefill_workload(seed, y_dtype):
    w = wl.make("prefill", seed, y_dtype=y_dtype, y0="randn" if seed else "zeros",
                shuffle_rows=seed == 2)
    y = run(w)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, f"prefill seed {seed} y {y_dtype}")


@pytest.mark.parametrize("r", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_ranks_and_input_types(r, dtype):
    lens = [130, 64, 257, 90]
    ra = torch.arange(4, dtype=torch.int32).repeat_interleave(torch.tensor(lens))
    w = wl.draw(int(sum(lens)), 5, 1024, 1032, r, ra, dtype=dtype, y_dtype=torch.float32,
                y0="randn", seed=r, scale=0.75)
    y = run(w)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, f"r={r} {dtype}")


def test_short_and_long_segments_in_one_call():
    # lengths straddle the 64-row threshold; ids unsorted in storage; one
    # long segment without an adapter
    lens = [3, 70, 1, 200, 64, 63, 129, 5, 80]
    ids = [0, 1, 2, 3, 4, 5, 6, 7, -1]
    ra = torch.tensor(ids, dtype=torch.int32).repeat_interleave(torch.tensor(lens))
    g = torch.Generator().manual_seed(3)
    ra = ra[torch.randperm(ra.numel(), generator=g)]
    w = wl.draw(ra.numel(), 8, 1536, 520, 64, ra, dtype=torch.bfloat16, y_dtype=torch.float32,
                y0="randn", seed=9, scale=1.5)
    y_dev = run(w)
    y_host = run(w, host_meta=True)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y_dev, ref, "device metadata")
    assert torch.equal(y_dev, y_host)
    untouched = (ra == -1).nonzero().flatten()
    assert torch.equal(y_dev[untouched].cpu(), w.Y0[untouched])


def test_split_between_cuda_and_tensor_cores():
    # decode rows (40 one-row segments) next to two long segments: segments
    # average under 8 rows, so the long ones go to the tensor cores and the
    # short ones to the CUDA-core kernel in the same call
    lens = [1] * 40 + [100, 80]
    ids = list(range(40)) + [40, 41]
    ra = torch.tensor(ids, dtype=torch.int32).repeat_interleave(torch.tensor(lens))
    g = torch.Generator().manual_seed(11)
    ra = ra[torch.randperm(ra.numel(), generator=g)]
    w = wl.draw(ra.numel(), 42, 1024, 776, 64, ra, dtype=torch.bfloat16, y_dtype=torch.float32,
                y0="randn", seed=12, scale=0.75)
    y_dev = run(w)
    y_host = run(w, host_meta=True)
    assert sg().sgmv_last_launch_count() == 3  # CUDA-core + tensor-core shrink + expand
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y_dev, ref, "split batch")
    assert torch.equal(y_dev, y_host)


@pytest.mark.parametrize("H1,H2", [(4104, 11016), (64, 136), (11008, 4096), (192, 8)])
def test_ragged_dims(H1, H2):
    lens = [150, 66]
    ra = torch.tensor([1, 0], dtype=torch.int32).repeat_interleave(torch.tensor(lens))
    w = wl.draw(216, 2, H1, H2, 64, ra, dtype=torch.bfloat16, y_dtype=torch.float32, y0="randn",
                seed=H1)
    y = run(w)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, f"H1={H1} H2={H2}")


def test_claimed_blocks_with_a_reused_workspace():
    """fp32 y: the last part of the expand's work is claimed at run time from
    a counter in the workspace, zeroed by each call's shrink kernel.  Three
    calls on one workspace, back to back: every call updates every block once
    (the oracle's result, and bit for bit the same y each time, whichever CTA
    took a block)."""
    w = wl.make("prefill", 1, y_dtype=torch.float32, y0="randn")
    X, A, B = w.X.to(DEV), w.A.to(DEV), w.B.to(DEV)
    perm, seg_ptr, idx, _ = sg().sgmv_build_segments_device(w.row_adapter.to(DEV), w.L)
    ws = torch.full((sg().sgmv_workspace_bytes(w.T, w.H1, w.H2, w.r),), 0x7f, dtype=torch.uint8,
                    device=DEV)  # the counter starts as garbage
    ys = [w.Y0.to(DEV).clone() for _ in range(3)]
    for y in ys:
        sg().sgmv_apply(y, X, A, B, seg_ptr, idx, w.scale, perm=perm, workspace=ws)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(ys[0], ref, "first call")
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])


@pytest.mark.parametrize("y_dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("H2", [1000, 4096])
def test_runs_cross_tiles(y_dtype, H2):
    """The expand's CTAs take equal weighted shares of the (tile, column
    block) line, so most runs end inside one tile and go on into the next:
    tiles of 128, 77, 5, 64 and 128 + 1 rows (shuffled rows), every block
    updated exactly once, each piece with its own rows and adapter."""
    lens = [205, 5, 64, 129]
    ra = torch.tensor([3, 0, 2, 1], dtype=torch.int32).repeat_interleave(torch.tensor(lens))
    g = torch.Generator().manual_seed(21)
    ra = ra[torch.randperm(len(ra), generator=g)]
    w = wl.draw(len(ra), 4, 256, H2, 64, ra, dtype=torch.float16, y_dtype=y_dtype, y0="randn",
                seed=H2)
    y = run(w)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, f"H2={H2} y {y_dtype}")


@pytest.mark.parametrize("y_dtype", [torch.float32, torch.bfloat16])
def test_more_tiles_than_sms(y_dtype):
    """More 128-row tiles than SMs: the expand's grid is a multiple of the SM
    count and its CTAs are dealt to tiles by weight; every (tile, column
    block) must be updated exactly once, for full and ragged tiles alike."""
    nsm = torch.cuda.get_device_properties(DEV).multi_processor_count
    g = torch.Generator().manual_seed(11)
    lens = []
    while sum((n + 127) // 128 for n in lens) <= nsm + 40:
        lens.append(int(torch.randint(129, 520, (1,), generator=g)))
    L = len(lens)
    ra = torch.arange(L, dtype=torch.int32).repeat_interleave(torch.tensor(lens))
    w = wl.draw(int(sum(lens)), L, 128, 264, 64, ra, dtype=torch.bfloat16, y_dtype=y_dtype,
                y0="randn", seed=12)
    y = run(w)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y, ref, f"{sum((n + 127) // 128 for n in lens)} tiles, y {y_dtype}")


def test_tensor_and_cuda_core_paths_agree():
    w = wl.make("prefill", 5, y0="randn")
    y_tc = run(w, ws=True)
    y_cc = run(w, ws=False)
    check_error_word(0)
    ref, *_ = oracle_apply_rows(w)
    assert_close(y_tc, ref, "tensor cores")
    assert_close(y_cc, ref, "CUDA cores")


def test_bad_adapter_in_long_segment_is_reported():
    lens = [100, 90]
    ra = torch.tensor([0, 1], dtype=torch.int32).repeat_interleave(torch.tensor(lens))
    w = wl.draw(190, 2, 512, 256, 64, ra, dtype=torch.bfloat16, y_dtype=torch.float32,
                y0="randn", seed=4)
    y = w.Y0.to(DEV).clone()
    seg_ptr = torch.tensor([0, 100, 190], dtype=torch.int32, device=DEV)
    idx = torch.tensor([0, 9], dtype=torch.int32, device=DEV)
    sg().sgmv_apply(y, w.X.to(DEV), w.A.to(DEV), w.B.to(DEV), seg_ptr, idx, w.scale,
                    workspace=workspace(w))
    check_error_word(4)
    assert torch.equal(y[100:].cpu(), w.Y0[100:])
    ref = oracle.sgmv_apply(w.Y0, w.X, w.A, w.B, [0, 100, 190], [0, -1], w.scale)
    assert_close(y, ref, "segment before the bad one")


def test_workspace_too_small_is_rejected():
    w = wl.draw(128, 1, 256, 256, 64, torch.zeros(128, dtype=torch.int32),
                dtype=torch.bfloat16)
    y = w.Y0.to(DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(sg().SgmvError) as e:
        sg().sgmv_apply(y, w.X.to(DEV), w.A.to(DEV), w.B.to(DEV),
                        torch.tensor([0, 128], dtype=torch.int32, device=DEV),
                        torch.tensor([0], dtype=torch.int32, device=DEV), 1.0, workspace=ws)
    assert e.value.status == 6
