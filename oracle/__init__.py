"""fp64 CPU oracle for SGMV (Segmented Gather Matrix-Vector multiplication).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
path (``rank_gemv_gb300``) never imports it, and this package imports nothing
from the product.

The arithmetic lives in ``sgmv_oracle.c`` (plain C, double precision, sums in
index order); this module compiles it with gcc on first use and marshals numpy
arrays.  What each function computes and which page passage it follows is
documented in that file.  Inputs are widened exactly from fp16 / bf16 / fp32 to
float64 by :func:`widen` before they reach the C code.

``Oracle(libpath)`` wraps one compiled library; the module-level functions use
the default build.  Tests that check the pins against deliberately broken
variants compile a modified copy of the C source and wrap it the same way.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "sgmv_oracle.c"
_BUILD_DIR = _HERE / "_build"

# -ffp-contract=off keeps a*b+c as two roundings on every host (gcc contracts
# to fused multiply-add by default on aarch64), so x86 and Arm hosts agree.
CFLAGS = ["-O2", "-std=c11", "-shared", "-fPIC", "-ffp-contract=off"]

_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)


def compile_source(src_text: str, out_dir: Path | None = None) -> Path:
    """Compile C source text into a shared library; returns its path.

    The library name carries a hash of the source, so a changed source is
    rebuilt and an unchanged one is reused.
    """
    out_dir = Path(out_dir) if out_dir is not None else _BUILD_DIR
    out_dir.mkdir(parents=True, exist_ok=True)
    digest = hashlib.sha1(src_text.encode()).hexdigest()[:12]
    lib = out_dir / f"liboracle_{digest}.so"
    if lib.exists():
        return lib
    src = out_dir / f"oracle_{digest}.c"
    src.write_text(src_text)
    tmp = out_dir / f".liboracle_{digest}.{os.getpid()}.so"
    subprocess.run(["gcc", *CFLAGS, "-o", str(tmp), str(src)], check=True)
    os.replace(tmp, lib)
    return lib


def build() -> Path:
    """Compile the oracle library from ``sgmv_oracle.c`` (idempotent)."""
    return compile_source(SOURCE.read_text())


def widen(t) -> np.ndarray:
    """Exact widening of a torch tensor or array to a C-contiguous float64 array."""
    if hasattr(t, "detach"):
        import torch

        return np.ascontiguousarray(t.detach().to("cpu", torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr_i32(a):
    return None if a is None else a.ctypes.data_as(_i32p)


class Oracle:
    """One compiled oracle library."""

    def __init__(self, libpath: str | os.PathLike):
        lib = ctypes.CDLL(str(libpath))
        lib.oracle_build_segments.restype = ctypes.c_int
        lib.oracle_build_segments.argtypes = [_i32p, ctypes.c_int32, ctypes.c_int32,
                                              _i32p, _i32p, _i32p, _i32p]
        lib.oracle_sgmv_shrink.restype = None
        lib.oracle_sgmv_shrink.argtypes = [_f64p, _f64p, _f64p, _i32p, _i32p, _i32p,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
        lib.oracle_sgmv_expand.restype = None
        lib.oracle_sgmv_expand.argtypes = [_f64p, _f64p, _f64p, ctypes.c_double, _i32p,
                                           _i32p, _i32p, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32]
        lib.oracle_sgmv_apply.restype = ctypes.c_int
        lib.oracle_sgmv_apply.argtypes = [_f64p, _f64p, _f64p, _f64p, ctypes.c_double,
                                          _i32p, _i32p, _i32p, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32]
        lib.oracle_fused_linear_lora.restype = ctypes.c_int
        lib.oracle_fused_linear_lora.argtypes = [_f64p, _f64p, _f64p, _f64p, _f64p,
                                                 ctypes.c_double, _i32p, _i32p, _i32p,
                                                 ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32]
        self._lib = lib
        self.path = str(libpath)

    # -- segment metadata -------------------------------------------------
    def build_segments(self, row_adapter, L: int):
        """Stable grouping of rows by adapter id -> (perm, seg_ptr, idx) int32 arrays."""
        ra = _i32(row_adapter).reshape(-1)
        T = ra.shape[0]
        perm = np.zeros(max(T, 1), np.int32)
        seg_ptr = np.zeros(max(T, 1) + 1, np.int32)
        idx = np.zeros(max(T, 1), np.int32)
        S = ctypes.c_int32(0)
        rc = self._lib.oracle_build_segments(_ptr_i32(ra), T, int(L), _ptr_i32(perm),
                                             _ptr_i32(seg_ptr), _ptr_i32(idx),
                                             ctypes.byref(S))
        if rc != 0:
            raise ValueError("adapter id outside [-1, L)")
        s = S.value
        return perm[:T].copy(), seg_ptr[: s + 1].copy(), idx[:s].copy()

    # -- SGMV -------------------------------------------------------------
    @staticmethod
    def _meta(seg_ptr, idx, perm, T):
        seg_ptr = _i32(seg_ptr).reshape(-1)
        idx = _i32(idx).reshape(-1)
        S = idx.shape[0]
        if seg_ptr.shape[0] != S + 1:
            raise ValueError("seg_ptr must have S+1 entries")
        if S and (seg_ptr[0] < 0 or seg_ptr[-1] > T or np.any(np.diff(seg_ptr) < 0)):
            raise ValueError("seg_ptr must be non-decreasing inside [0, T]")
        p = None
        if perm is not None:
            p = _i32(perm).reshape(-1)
            if p.shape[0] < (seg_ptr[-1] if S else 0):
                raise ValueError("perm too short")
            if p.size and (p.min() < 0 or p.max() >= T):
                raise ValueError("perm entry outside [0, T)")
        return seg_ptr, idx, S, p

    def sgmv_shrink(self, X, A, seg_ptr, idx, perm=None):
        """v[T, r] (float64), zero where no segment covers a position."""
        X = widen(X)
        A = widen(A)
        T, H1 = X.shape
        L, H1a, r = A.shape
        assert H1a == H1
        seg_ptr, idx, S, p = self._meta(seg_ptr, idx, perm, T)
        if S and (idx.max() >= L or idx.min() < -1):
            raise ValueError("adapter id outside [-1, L)")
        v = np.zeros((T, r), np.float64)
        self._lib.oracle_sgmv_shrink(v.ctypes.data_as(_f64p), X.ctypes.data_as(_f64p),
                                     A.ctypes.data_as(_f64p), _ptr_i32(p), _ptr_i32(seg_ptr),
                                     _ptr_i32(idx), S, H1, r)
        return v

    def sgmv_expand(self, Y, v, B, seg_ptr, idx, scale, perm=None):
        """Returns a float64 copy of Y with the expand step added."""
        Y = widen(Y).copy()
        v = widen(v)
        B = widen(B)
        T, H2 = Y.shape
        L, r, H2b = B.shape
        assert H2b == H2 and v.shape == (T, r)
        seg_ptr, idx, S, p = self._meta(seg_ptr, idx, perm, T)
        if S and (idx.max() >= L or idx.min() < -1):
            raise ValueError("adapter id outside [-1, L)")
        self._lib.oracle_sgmv_expand(Y.ctypes.data_as(_f64p), v.ctypes.data_as(_f64p),
                                     B.ctypes.data_as(_f64p), float(scale), _ptr_i32(p),
                                     _ptr_i32(seg_ptr), _ptr_i32(idx), S, H2, r)
        return Y

    def sgmv_apply(self, Y, X, A, B, seg_ptr, idx, scale, perm=None, *, widened=False):
        """Returns a float64 copy of Y + scale * SGMV delta.

        With ``widened=True`` the inputs must already be C-contiguous float64
        arrays (Y is still copied); the benchmark uses this to time the C code
        without re-widening the stacked weights on every call.
        """
        if not widened:
            Y, X, A, B = widen(Y), widen(X), widen(A), widen(B)
        Y = Y.copy()
        T, H2 = Y.shape
        T2, H1 = X.shape
        L, H1a, r = A.shape
        assert T2 == T and H1a == H1 and B.shape == (L, r, H2)
        seg_ptr, idx, S, p = self._meta(seg_ptr, idx, perm, T)
        if S and (idx.max() >= L or idx.min() < -1):
            raise ValueError("adapter id outside [-1, L)")
        rc = self._lib.oracle_sgmv_apply(Y.ctypes.data_as(_f64p), X.ctypes.data_as(_f64p),
                                         A.ctypes.data_as(_f64p), B.ctypes.data_as(_f64p),
                                         float(scale), _ptr_i32(p), _ptr_i32(seg_ptr),
                                         _ptr_i32(idx), S, T, H1, H2, r)
        if rc != 0:
            raise MemoryError("oracle temporary allocation failed")
        return Y


    def fused_linear_lora(self, X, W, A, B, seg_ptr, idx, scale, perm=None):
        """float64 Y[T, H2] = X.W + scale * SGMV delta (the base output alone
        on rows of no adapter); W is [H1, H2]."""
        X, W, A, B = widen(X), widen(W), widen(A), widen(B)
        T, H1 = X.shape
        H1w, H2 = W.shape
        L, H1a, r = A.shape
        assert H1w == H1 and H1a == H1 and B.shape == (L, r, H2)
        seg_ptr, idx, S, p = self._meta(seg_ptr, idx, perm, T)
        if S and (idx.max() >= L or idx.min() < -1):
            raise ValueError("adapter id outside [-1, L)")
        Y = np.zeros((T, H2), np.float64)
        rc = self._lib.oracle_fused_linear_lora(Y.ctypes.data_as(_f64p), X.ctypes.data_as(_f64p),
                                                W.ctypes.data_as(_f64p), A.ctypes.data_as(_f64p),
                                                B.ctypes.data_as(_f64p), float(scale),
                                                _ptr_i32(p), _ptr_i32(seg_ptr), _ptr_i32(idx),
                                                S, T, H1, H2, r)
        if rc != 0:
            raise MemoryError("oracle temporary allocation failed")
        return Y


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def build_segments(row_adapter, L):
    return default().build_segments(row_adapter, L)


def sgmv_shrink(X, A, seg_ptr, idx, perm=None):
    return default().sgmv_shrink(X, A, seg_ptr, idx, perm)


def sgmv_expand(Y, v, B, seg_ptr, idx, scale, perm=None):
    return default().sgmv_expand(Y, v, B, seg_ptr, idx, scale, perm)


def sgmv_apply(Y, X, A, B, seg_ptr, idx, scale, perm=None, *, widened=False):
    return default().sgmv_apply(Y, X, A, B, seg_ptr, idx, scale, perm, widened=widened)


def fused_linear_lora(X, W, A, B, seg_ptr, idx, scale, perm=None):
    return default().fused_linear_lora(X, W, A, B, seg_ptr, idx, scale, perm)
