"""Shared helpers of the GPU parity tests: tolerance, runs of the CUDA path
through the C ABI, and the oracle's reference for the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def tolerance(ref: np.ndarray, y_dtype) -> np.ndarray:
    """Per-element bound on |Y_gpu - Y_ref|.

    The bound is max|dY| <= 1e-2 * RMS(Y_ref).  A bf16 output cannot meet it
    where |Y_ref| is large (half an ulp of bf16 is 2^-8 |Y|), so for bf16
    outputs half an ulp of the output at |Y_ref| is added per element.
    """
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bound = np.full(ref.shape, 1e-2 * rms)
    if y_dtype == torch.bfloat16:
        mag = np.maximum(np.abs(ref), np.finfo(np.float32).tiny)
        bound = bound + 0.5 * np.exp2(np.floor(np.log2(mag)) - 7)
    return bound


def assert_close(y_gpu: torch.Tensor, ref: np.ndarray, what: str = ""):
    y = y_gpu.detach().double().cpu().numpy()
    assert y.shape == ref.shape
    err = np.abs(y - ref)
    bound = tolerance(ref, y_gpu.dtype)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"gpu={y[i]!r} ref={ref[i]!r} bound={bound[i]:.3e}")


def device_grouping(row_adapter: torch.Tensor, L: int):
    from rank_gemv_gb300 import sgmv

    return sgmv.sgmv_build_segments_device(row_adapter.to("cuda"), L)


def gpu_apply_rows(w, *, use_host_meta=False):
    """The benchmarked configuration: group rows on the device, then the fused
    update with the permutation.  Returns (y, perm, seg_ptr, idx, S)."""
    from rank_gemv_gb300 import sgmv

    dev = torch.device("cuda")
    y = w.Y0.to(dev).clone()
    if use_host_meta:
        perm, seg_ptr, idx = sgmv.sgmv_build_segments(w.row_adapter, w.L)
        S = torch.tensor([idx.numel()], dtype=torch.int32)
        sgmv.sgmv_apply(y, w.X.to(dev), w.A.to(dev), w.B.to(dev), seg_ptr.to(dev), idx.to(dev),
                        w.scale, perm=perm.to(dev), seg_ptr_host=seg_ptr)
        return y, perm, seg_ptr, idx, S
    perm, seg_ptr, idx, S = device_grouping(w.row_adapter, w.L)
    sgmv.sgmv_apply(y, w.X.to(dev), w.A.to(dev), w.B.to(dev), seg_ptr, idx, w.scale, perm=perm)
    return y, perm, seg_ptr, idx, S


def oracle_apply_rows(w):
    perm, seg_ptr, idx = oracle.build_segments(w.row_adapter, w.L)
    ref = oracle.sgmv_apply(w.Y0, w.X, w.A, w.B, seg_ptr, idx, w.scale, perm=perm)
    return ref, perm, seg_ptr, idx


def check_error_word(expected=0):
    from rank_gemv_gb300 import sgmv

    got = sgmv.sgmv_get_device_error()
    assert got == expected, f"device error word {got}, expected {expected}"
