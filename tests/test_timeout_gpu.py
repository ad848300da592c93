"""Device-side timeout reporting of the streaming kernel.

Every wait inside a kernel is bounded; when one runs out, the kernel sets
SGMV_ERR_TIMEOUT in the device error word instead of trapping ("Punica: when
LoRA fine-tuned models need multi-tenant serving", omica.com.cn article, §5.2:
a shape mismatch shows up as an illegal memory access, so the library
reports device-side problems as status codes and keeps the context usable).

A real timeout needs a copy that never lands, which cannot be made safely on
a shared GPU.  sgmv_debug_inject_wait_timeout makes each compute thread's
first wait for a staged chunk take the timeout path without polling; the
rest of that path is the one a real timeout runs: the error word is set, the
chunk is awaited once more with the full limit (so every copy lands before
the CTA moves on and the kernel ends normally) and the thread stops writing
y.  The tests check the status, that no output was written, and that the
next call on the same context is correct.
"""
import pytest
import torch

from rank_gemv_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, check_error_word, oracle_apply_rows

pytestmark = pytest.mark.gpu


def _run(w, inject):
    from rank_gemv_gb300 import sgmv

    dev = torch.device("cuda")
    smax = sgmv.sgmv_max_segments(w.T, w.L)
    meta = (torch.empty(w.T, dtype=torch.int32, device=dev),
            torch.empty(smax + 1, dtype=torch.int32, device=dev),
            torch.empty(smax, dtype=torch.int32, device=dev),
            torch.empty(1, dtype=torch.int32, device=dev))
    y = w.Y0.to(dev).clone()
    sgmv.sgmv_debug_inject_wait_timeout(inject)
    try:
        sgmv.sgmv_apply_rows(y, w.X.to(dev), w.A.to(dev), w.B.to(dev), w.row_adapter.to(dev),
                             w.scale, out=meta)
    finally:
        sgmv.sgmv_debug_inject_wait_timeout(False)
    return y


@pytest.mark.parametrize("name,T", [("decode-distinct", None), ("custom", 100)])
def test_injected_timeout_is_reported_and_the_context_stays_usable(name, T):
    """decode-distinct runs the one-launch grouped form (32 rows); 100 rows on
    100 adapters run the grouping kernel, then the streaming kernel on the
    device metadata."""
    from rank_gemv_gb300 import sgmv

    if T is None:
        w = wl.make(name, 5, y0="randn", shuffle_rows=True)
    else:
        g = torch.Generator().manual_seed(T)
        ids = torch.randperm(T, generator=g).to(torch.int32)
        w = wl.draw(T, T, 1024, 2048, 16, ids, seed=T, y0="randn")
    check_error_word(0)
    y = _run(w, True)
    assert sgmv.sgmv_get_device_error() == 7  # SGMV_ERR_TIMEOUT, and the word is cleared
    # every compute thread took the timeout path before its first y write
    assert torch.equal(y.cpu(), w.Y0)
    y2 = _run(w, False)
    check_error_word(0)
    assert_close(y2, oracle_apply_rows(w)[0], f"{name}: the call after the reported timeout")


def test_injected_timeout_in_a_multi_problem_launch():
    """Three problems on 100 rows in one launch of the multi-problem
    instantiation: the injected timeout is reported, no y is written, and the
    next launch is correct."""
    import oracle
    from rank_gemv_gb300 import sgmv

    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(7)
    ids = torch.randint(0, 12, (100,), generator=g, dtype=torch.int32)
    ws = [wl.draw(100, 12, 1024, 520, 16, ids, seed=70 + k, y0="randn") for k in range(3)]
    perm, seg_ptr, idx, _ = sgmv.sgmv_build_segments_device(ids.to(dev), 12)
    S = sgmv.sgmv_max_segments(100, 12)
    args = ([w.X.to(dev) for w in ws], [w.A.to(dev) for w in ws], [w.B.to(dev) for w in ws])

    def run(inject):
        ys = [w.Y0.to(dev) for w in ws]
        sgmv.sgmv_debug_inject_wait_timeout(inject)
        try:
            sgmv.sgmv_apply_multi(ys, *args, seg_ptr, idx, 1.0, perm=perm, S=S)
            assert sgmv.load_library().sgmv_last_launch_count() == 1
        finally:
            sgmv.sgmv_debug_inject_wait_timeout(False)
        return ys

    check_error_word(0)
    ys = run(True)
    assert sgmv.sgmv_get_device_error() == 7
    for y, w in zip(ys, ws):
        assert torch.equal(y.cpu(), w.Y0)
    ys = run(False)
    check_error_word(0)
    o_perm, o_seg, o_idx = oracle.build_segments(ids, 12)
    for k, (y, w) in enumerate(zip(ys, ws)):
        ref = oracle.sgmv_apply(w.Y0, w.X, w.A, w.B, o_seg, o_idx, 1.0, perm=o_perm)
        assert_close(y, ref, f"problem {k} after the reported timeout")
