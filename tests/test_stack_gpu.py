"""Full-size llama7b-stack workload (32 layers x 7 projections, 128 decode rows
on 128 adapters, about 10 GB of stacked adapters) in the benchmark's launch
configuration: one device grouping, then per layer q+k+v, o, gate+up and
down as one sgmv_apply_multi launch each.  Five
projections are checked against the oracle element by element, and three
rows of every one of the 224 projections (each row against the oracle on
that row and its adapter alone)."""
import pytest
import torch

import oracle
from rank_gemv_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, check_error_word

pytestmark = pytest.mark.gpu

SAMPLES = [(0, 0), (9, 3), (17, 4), (24, 5), (31, 6)]  # (layer, projection)


def test_llama7b_stack_sampled_projections():
    from rank_gemv_gb300 import build, sgmv

    build.build()
    dev = torch.device("cuda")
    seed = 0
    projs = [wl.stack_projection(seed, layer, p, device=dev)
             for layer in range(wl.LLAMA7B_LAYERS) for p in range(len(wl.LLAMA7B_PROJ))]
    ra = wl.stack_row_adapter(128)
    perm, seg_ptr, idx, S = sgmv.sgmv_build_segments_device(ra.to(dev), 128)
    smax = sgmv.sgmv_max_segments(128, 128)
    n_proj = len(wl.LLAMA7B_PROJ)
    for layer in range(wl.LLAMA7B_LAYERS):
        for g in ([0, 1, 2], [3], [4, 5], [6]):
            pr = [projs[layer * n_proj + k] for k in g]
            sgmv.sgmv_apply_multi([p[3] for p in pr], [p[0] for p in pr],
                                  [p[1] for p in pr], [p[2] for p in pr], seg_ptr, idx, 1.0,
                                  perm=perm, S=smax)
            assert sgmv.load_library().sgmv_last_launch_count() == 1
    check_error_word(0)
    o_perm, o_seg, o_idx = oracle.build_segments(ra, 128)
    for layer, p in SAMPLES:
        X, A, B, Y = projs[layer * n_proj + p]
        Y0 = torch.zeros(Y.shape, dtype=torch.float16)
        ref = oracle.sgmv_apply(Y0, X, A, B, o_seg, o_idx, 1.0, perm=o_perm)
        assert_close(Y, ref, f"layer {layer} proj {wl.LLAMA7B_PROJ[p][0]}")
    one = (torch.tensor([0, 1], dtype=torch.int32), torch.tensor([0], dtype=torch.int32))
    for k, (X, A, B, Y) in enumerate(projs):
        layer, p = divmod(k, n_proj)
        for t in ((7 * k + 3) % 128, (13 * k + 64) % 128, (29 * k + 101) % 128):
            a = int(ra[t])
            ref = oracle.sgmv_apply(torch.zeros((1, Y.shape[1]), dtype=torch.float16),
                                    X[t:t + 1].cpu(), A[a:a + 1].cpu(), B[a:a + 1].cpu(),
                                    one[0], one[1], 1.0)
            assert_close(Y[t:t + 1], ref, f"layer {layer} proj {wl.LLAMA7B_PROJ[p][0]} row {t}")
    del projs
    torch.cuda.empty_cache()
