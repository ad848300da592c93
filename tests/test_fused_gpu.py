"""The fused LoRA layer y = x W + scale * (x A[a]) B[a] (sgmv_fused_linear_lora)
against the oracle's fused layer, element by element.

The layer follows "Punica: when LoRA fine-tuned models need multi-tenant
serving" (omica.com.cn article, §2.1: y = xW + xAB) with the adapter update of
SGMV, fused into the base linear layer as "How to deploy several LoRA adapters
without reloading the base model (Punica, S-LoRA)?" (aivaro.ru, §3.2, "Fused
Kernel") describes.  Cases: the Llama-2-7B q projection with 128 decode rows
on 128 adapters (sampled rows), batches of 1 to 128 rows (ragged against the
16-row blocks), shuffled rows, rows of no adapter, adapters shared by long
segments, ragged H1 / H2, ranks 8 to 64, every input / output type pair, no
segment at all, and the grouping straight from sgmv_build_segments_device
(padded with empty segments).
"""
import numpy as np
import pytest
import torch

import oracle
from rank_gemv_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, check_error_word

pytestmark = pytest.mark.gpu

F16, BF16, F32 = torch.float16, torch.bfloat16, torch.float32


def _problem(T, L, H1, H2, r, ids, *, dtype=F16, y_dtype=None, seed=0, scale=1.0):
    w = wl.draw(T, L, H1, H2, r, ids, dtype=dtype, y_dtype=y_dtype, seed=seed, y0="randn",
                scale=scale)
    W = wl.base_weight(H1, H2, dtype=dtype, seed=seed + 101)
    return w, W


def _run(w, W, *, device_grouping=True):
    from rank_gemv_gb300 import sgmv

    dev = torch.device("cuda")
    if device_grouping:
        perm, seg_ptr, idx, _ = sgmv.sgmv_build_segments_device(w.row_adapter.to(dev), w.L)
    else:
        perm, seg_ptr, idx = (t.to(dev) for t in sgmv.sgmv_build_segments(w.row_adapter, w.L))
    y = torch.full((w.T, w.H2), 7.0, dtype=w.y_dtype, device=dev)  # overwritten
    sgmv.sgmv_fused_linear_lora(y, w.X.to(dev), W.to(dev), w.A.to(dev), w.B.to(dev), seg_ptr,
                                idx, w.scale, perm=perm)
    assert sgmv.sgmv_last_launch_count() == 3  # shrink, v tiles, fused layer
    check_error_word(0)
    return y


def _ref(w, W, rows=None):
    ra = w.row_adapter if rows is None else w.row_adapter[rows]
    X = w.X if rows is None else w.X[rows]
    perm, seg_ptr, idx = oracle.build_segments(ra, w.L)
    return oracle.fused_linear_lora(X, W, w.A, w.B, seg_ptr, idx, w.scale, perm=perm)


def test_llama7b_q_decode_128_rows_on_128_adapters():
    """4096 -> 4096, r = 16, fp16: every row its own adapter, rows shuffled;
    ten sampled rows checked against the oracle (the whole batch against the
    base product plus the SGMV path)."""
    from rank_gemv_gb300 import sgmv

    g = torch.Generator().manual_seed(3)
    ids = torch.randperm(128, generator=g).to(torch.int32)
    w, W = _problem(128, 128, 4096, 4096, 16, ids, seed=3)
    y = _run(w, W)
    rows = torch.tensor([0, 1, 15, 16, 31, 64, 77, 100, 126, 127])
    assert_close(y[rows.cuda()], _ref(w, W, rows), "q projection, sampled rows")
    # every row: the same layer through cuBLAS x W (fp32) and SGMV on fp32 y
    dev = torch.device("cuda")
    y32 = (w.X.to(dev).float() @ W.to(dev).float()).contiguous()
    sgmv.sgmv_apply_rows(y32, w.X.to(dev), w.A.to(dev), w.B.to(dev), w.row_adapter.to(dev), 1.0,
                         out=sgmv.sgmv_build_segments_device(w.row_adapter.to(dev), w.L))
    assert_close(y, y32.double().cpu().numpy(), "q projection, all rows vs x W + SGMV")


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 33, 64, 100, 127, 128])
def test_batch_sizes(T):
    g = torch.Generator().manual_seed(T)
    ids = torch.randint(-1, 6, (T,), generator=g, dtype=torch.int32)
    w, W = _problem(T, 6, 512, 384, 16, ids, seed=T)
    assert_close(_run(w, W), _ref(w, W), f"T={T}")


@pytest.mark.parametrize("H1,H2", [(64, 64), (136, 200), (1000, 520), (4096, 11008 // 8)])
def test_ragged_dimensions(H1, H2):
    g = torch.Generator().manual_seed(H1 + H2)
    ids = torch.randint(-1, 5, (40,), generator=g, dtype=torch.int32)
    w, W = _problem(40, 5, H1, H2, 16, ids, seed=H1)
    assert_close(_run(w, W), _ref(w, W), f"H1={H1} H2={H2}")


@pytest.mark.parametrize("r", [1, 8, 16, 24, 32, 64])
def test_ranks(r):
    g = torch.Generator().manual_seed(r)
    ids = torch.randint(0, 9, (48,), generator=g, dtype=torch.int32)
    w, W = _problem(48, 9, 768, 640, r, ids, seed=r, scale=0.5)
    assert_close(_run(w, W), _ref(w, W), f"r={r}")


@pytest.mark.parametrize("scale", [0.0, -2.0, 1e-3])
def test_scale_values(scale):
    """scale multiplies the adapter term only: 0 gives x W exactly, a negative
    scale flips the term's sign (v's hi / lo halves carry the sign), a small
    one leaves the term below the base product's rounding."""
    g = torch.Generator().manual_seed(7)
    ids = torch.randint(-1, 6, (40,), generator=g, dtype=torch.int32)
    w, W = _problem(40, 6, 512, 384, 16, ids, seed=11, scale=scale)
    assert_close(_run(w, W), _ref(w, W), f"scale {scale}")


@pytest.mark.parametrize("dtype,y_dtype", [(F16, F16), (F16, F32), (BF16, BF16), (BF16, F32),
                                           (F16, BF16), (BF16, F16)])
def test_types(dtype, y_dtype):
    g = torch.Generator().manual_seed(5)
    ids = torch.randint(-1, 4, (70,), generator=g, dtype=torch.int32)
    w, W = _problem(70, 4, 1024, 768, 32, ids, dtype=dtype, y_dtype=y_dtype, seed=5)
    assert_close(_run(w, W), _ref(w, W), f"{dtype} -> {y_dtype}")


def test_long_shared_segments_and_host_grouping():
    """Two adapters over 100 rows (segments of 60 and 40 spread over every
    16-row block), metadata from the host grouping (no padding)."""
    g = torch.Generator().manual_seed(9)
    ids = torch.tensor([0] * 60 + [3] * 40, dtype=torch.int32)[torch.randperm(100, generator=g)]
    w, W = _problem(100, 4, 2048, 1024, 64, ids, seed=9)
    assert_close(_run(w, W, device_grouping=False), _ref(w, W), "shared adapters")


def test_no_adapter_at_all_is_the_base_layer():
    from rank_gemv_gb300 import sgmv

    ids = torch.full((24,), -1, dtype=torch.int32)
    w, W = _problem(24, 2, 512, 256, 16, ids, seed=2)
    assert_close(_run(w, W), _ref(w, W), "every row without an adapter")
    # no segments: base product only (one kernel)
    dev = torch.device("cuda")
    y = torch.zeros((24, 256), dtype=F16, device=dev)
    empty = torch.zeros(1, dtype=torch.int32, device=dev)
    sgmv.sgmv_fused_linear_lora(y, w.X.to(dev), W.to(dev), w.A.to(dev), w.B.to(dev), empty,
                                empty[:0], 1.0)
    assert sgmv.sgmv_last_launch_count() == 1
    check_error_word(0)
    base = w.X.double().numpy() @ W.double().numpy()
    assert_close(y, base, "no segments")


def test_bad_adapter_id_is_reported_and_its_rows_get_the_base_product():
    from rank_gemv_gb300 import sgmv

    dev = torch.device("cuda")
    ids = torch.tensor([0, 1, 1, 0], dtype=torch.int32)
    w, W = _problem(4, 2, 256, 128, 16, ids, seed=4)
    perm, seg_ptr, idx = sgmv.sgmv_build_segments(w.row_adapter, w.L)
    idx_bad = idx.clone()
    idx_bad[1] = 5  # adapter 1's segment now names an adapter outside the pool
    y = torch.zeros((4, 128), dtype=F16, device=dev)
    sgmv.sgmv_fused_linear_lora(y, w.X.to(dev), W.to(dev), w.A.to(dev), w.B.to(dev),
                                seg_ptr.to(dev), idx_bad.to(dev), 1.0, perm=perm.to(dev))
    assert sgmv.sgmv_get_device_error() == 4
    ref = _ref(w, W)
    base = w.X.double().numpy() @ W.double().numpy()
    for t in range(4):
        want = ref[t] if int(ids[t]) == 0 else base[t]
        assert_close(y[t:t + 1], want[None], f"row {t}")
