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
