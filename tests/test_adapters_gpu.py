"""On-demand adapter loading: SGMV on the slots an AdapterPool filled.

Two projections (512 -> 264 and 264 -> 512, r = 16) with 4 slots serve
batches over 6 adapters, so adapters are loaded (by the gather kernel, or by
copy-engine transfers), evicted and reloaded.  After
each batch: every resident slot holds its adapter's weights bit for bit, and
SGMV on the slots gives the oracle's result computed directly from each row's
adapter weights.
"""
import pytest
import torch

import oracle
from rank_gemv_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, check_error_word

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
PROJ = [(512, 264), (264, 512)]
R, L, NAMES = 16, 4, ["a", "b", "c", "d", "e", "f"]


def host_adapters():
    g = torch.Generator().manual_seed(5)
    out = {}
    for n in NAMES:
        out[n] = [((torch.randn(h1, R, generator=g) * h1 ** -0.5).half().pin_memory(),
                   (torch.randn(R, h2, generator=g) * R ** -0.5).half().pin_memory())
                  for h1, h2 in PROJ]
    return out


@pytest.mark.parametrize("gather", [True, False])
def test_batches_through_loaded_slots(gather):
    from rank_gemv_gb300 import build, sgmv
    from rank_gemv_gb300.adapters import AdapterPool

    build.build()
    sgmv.load_library()
    weights = host_adapters()
    pools = [(torch.full((L, h1, R), float("nan"), dtype=torch.half, device=DEV),
              torch.full((L, R, h2), float("nan"), dtype=torch.half, device=DEV))
             for h1, h2 in PROJ]
    pool = AdapterPool(pools, source=lambda n: weights[n], gather=gather)
    batches = [["a", "b", "c", "a"], ["d", "e", "a", "a", "b"], ["f", "b", "b", "c"],
               ["a", "f"], ["e", "d", "c", "b"]]
    g = torch.Generator().manual_seed(9)
    for names in batches:
        slots = pool.slots_for(names)
        ra = torch.tensor(slots, dtype=torch.int32)
        ids = torch.tensor([NAMES.index(n) for n in names], dtype=torch.int32)
        for p, (h1, h2) in enumerate(PROJ):
            X = torch.randn(len(names), h1, generator=g).half()
            Y0 = torch.randn(len(names), h2, generator=g).half()
            y = Y0.to(DEV)
            sgmv.sgmv_apply_rows(y, X.to(DEV), pools[p][0], pools[p][1], ra.to(DEV), 0.5)
            A_all = torch.stack([weights[n][p][0] for n in NAMES])
            B_all = torch.stack([weights[n][p][1] for n in NAMES])
            perm, seg_ptr, idx = oracle.build_segments(ids, len(NAMES))
            ref = oracle.sgmv_apply(Y0, X, A_all, B_all, seg_ptr, idx, 0.5, perm=perm)
            assert_close(y, ref, f"batch {names}, projection {p}")
        check_error_word(0)
        torch.cuda.synchronize()
        for n, slot in pool.resident.items():
            for p in range(len(PROJ)):
                assert torch.equal(pools[p][0][slot].cpu(), weights[n][p][0])
                assert torch.equal(pools[p][1][slot].cpu(), weights[n][p][1])
    assert pool.loads > len(NAMES)  # some adapters were evicted and loaded again


def test_bad_arguments_are_refused():
    from rank_gemv_gb300 import sgmv

    A = torch.zeros(2, 64, 16, dtype=torch.half, device=DEV)
    B = torch.zeros(2, 16, 64, dtype=torch.half, device=DEV)
    a = torch.zeros(64, 16, dtype=torch.half)
    b = torch.zeros(16, 64, dtype=torch.half)
    with pytest.raises(sgmv.SgmvError) as e:
        sgmv.sgmv_load_adapter(A, B, 2, a, b)
    assert e.value.status == 1
    with pytest.raises(ValueError):
        sgmv.sgmv_load_adapter(A, B, 0, a[:32], b)
