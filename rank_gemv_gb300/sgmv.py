"""Thin ctypes binding of libsgmv.so (C ABI in include/sgmv.h).

Argument marshalling only: every step of SGMV runs in the library's CUDA
kernels.  Tensors are torch tensors (PyTorch provides device memory and the
current stream); each function passes their data pointers, sizes and
``torch.cuda.current_stream()`` to the C function of the same name and raises
:class:`SgmvError` on a non-zero status.  If the library has not been built
(``__graft_entry__.build()`` or ``python -m rank_gemv_gb300.build``), loading
it raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

LIB_PATH = Path(__file__).resolve().parent / "libsgmv.so"

SGMV_F16, SGMV_BF16, SGMV_F32 = 0, 1, 2
_DTYPES = {torch.float16: SGMV_F16, torch.bfloat16: SGMV_BF16, torch.float32: SGMV_F32}

STATUS = {0: "SGMV_OK", 1: "SGMV_ERR_INVALID_ARG", 2: "SGMV_ERR_UNSUPPORTED",
          3: "SGMV_ERR_ALIGNMENT", 4: "SGMV_ERR_BAD_INDEX", 5: "SGMV_ERR_CUDA",
          6: "SGMV_ERR_WORKSPACE", 7: "SGMV_ERR_TIMEOUT", 8: "SGMV_ERR_BAD_SEGMENTS"}

# Every function include/sgmv.h declares, with its ctypes signature.
_vp, _i32, _i32p = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)
_int, _f32, _sz = ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_vpp, _u64p = ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_uint64)
SIGNATURES = {
    "sgmv_status_string": (ctypes.c_char_p, [_int]),
    "sgmv_last_error_string": (ctypes.c_char_p, []),
    "sgmv_last_launch_count": (_int, []),
    "sgmv_max_segments": (_i32, [_i32, _i32]),
    "sgmv_build_segments": (_int, [_vp, _i32, _i32, _vp, _vp, _vp, _vp]),
    "sgmv_build_segments_device": (_int, [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "sgmv_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "sgmv_shrink": (_int, [_vp, _vp, _vp, _int, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                           _i32, _vp]),
    "sgmv_expand": (_int, [_vp, _int, _vp, _vp, _int, _f32, _vp, _vp, _vp, _i32, _vp, _i32,
                           _i32, _i32, _i32, _vp]),
    "sgmv_apply": (_int, [_vp, _int, _vp, _vp, _vp, _int, _f32, _vp, _vp, _vp, _i32, _vp, _i32,
                          _i32, _i32, _i32, _i32, _vp, _sz, _vp]),
    "sgmv_apply_rows": (_int, [_vp, _int, _vp, _vp, _vp, _int, _f32, _vp, _i32, _i32, _i32, _i32,
                               _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sgmv_apply_multi": (_int, [_i32, _vpp, _int, _vpp, _vpp, _vpp, _int, _f32, _vp, _vp, _vp,
                                _i32, _vp, _i32, _i32, _i32, _i32, _i32, _vp]),
    "sgmv_apply_noalloc": (_int, [_vp, _int, _vp, _vp, _vp, _int, _f32, _vp, _vp, _vp, _i32, _vp,
                                  _i32, _i32, _i32, _i32, _i32, _vp]),
    "sgmv_fused_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "sgmv_fused_linear_lora": (_int, [_vp, _int, _vp, _vp, _vp, _vp, _int, _f32, _vp, _vp, _vp,
                                      _i32, _i32, _i32, _i32, _i32, _i32, _vp, _sz, _vp]),
    "sgmv_load_adapter": (_int, [_vp, _vp, _int, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _vp]),
    "sgmv_copy_gather": (_int, [_i32, _vpp, _vpp, _u64p, _i32, _vp]),
    "sgmv_read_floor": (_int, [_vp, _sz, _i32, _i32, _i32, _i32, _i32, _int, _int, _i32p, _i32p,
                               _vp]),
    "sgmv_debug_inject_wait_timeout": (_int, [_int]),
    "sgmv_get_device_error": (_int, [_vp]),
}

_lib = None


class SgmvError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


def load_library(path: str | Path | None = None) -> ctypes.CDLL:
    """Load libsgmv.so (once) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path is not None else LIB_PATH
    if not p.exists():
        raise RuntimeError(f"{p} is not built: run __graft_entry__.build() first")
    lib = ctypes.CDLL(str(p))
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(rc: int, where: str):
    if rc != 0:
        detail = ""
        if rc == 5:
            detail = (load_library().sgmv_last_error_string() or b"").decode()
        raise SgmvError(rc, where, detail)


def _ptr(t):
    return None if t is None else t.data_ptr()


# pointer-array types for the multi-problem entry (P = 1 .. 4)
_PTR_ARRAYS = [None] + [ctypes.c_void_p * n for n in range(1, 5)]


def _stream(device):
    return torch.cuda.current_stream(device).cuda_stream


def _meta(t, name):
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous int32 tensor")
    return t


def _host_i32(a):
    if a is None:
        return None
    t = torch.as_tensor(a, dtype=torch.int32, device="cpu").contiguous()
    return t


def sgmv_status_string(status: int) -> str:
    return load_library().sgmv_status_string(status).decode()


def sgmv_last_launch_count() -> int:
    """Kernels launched by this thread's last launching call."""
    return int(load_library().sgmv_last_launch_count())


def sgmv_max_segments(T: int, L: int) -> int:
    return int(load_library().sgmv_max_segments(T, L))


def sgmv_workspace_bytes(T: int, H1: int, H2: int, r: int) -> int:
    return int(load_library().sgmv_workspace_bytes(T, H1, H2, r))


def sgmv_build_segments(row_adapter, L: int):
    """Host grouping -> (perm, seg_ptr, idx) as CPU int32 tensors."""
    ra = _host_i32(row_adapter).reshape(-1)
    T = ra.numel()
    perm = torch.empty(max(T, 1), dtype=torch.int32)
    seg_ptr = torch.empty(T + 1, dtype=torch.int32)
    idx = torch.empty(max(T, 1), dtype=torch.int32)
    S = ctypes.c_int32(0)
    _check(load_library().sgmv_build_segments(ra.data_ptr(), T, L, perm.data_ptr(),
                                              seg_ptr.data_ptr(), idx.data_ptr(),
                                              ctypes.addressof(S)), "sgmv_build_segments")
    s = S.value
    return perm[:T].clone(), seg_ptr[: s + 1].clone(), idx[:s].clone()


def sgmv_build_segments_device(row_adapter: torch.Tensor, L: int, out=None):
    """Device grouping -> (perm, seg_ptr, idx, S) device int32 tensors, padded to
    sgmv_max_segments(T, L) segments (S holds the real count on the device)."""
    ra = _meta(row_adapter, "row_adapter")
    T = ra.numel()
    smax = sgmv_max_segments(T, L)
    if out is None:
        dev = ra.device
        out = (torch.empty(max(T, 1), dtype=torch.int32, device=dev),
               torch.empty(smax + 1, dtype=torch.int32, device=dev),
               torch.empty(max(smax, 1), dtype=torch.int32, device=dev),
               torch.empty(1, dtype=torch.int32, device=dev))
    perm, seg_ptr, idx, S = out
    _check(load_library().sgmv_build_segments_device(
        ra.data_ptr(), T, L, perm.data_ptr(), seg_ptr.data_ptr(), idx.data_ptr(), S.data_ptr(),
        _stream(ra.device)), "sgmv_build_segments_device")
    return perm, seg_ptr, idx, S


def _nseg(idx, S):
    return idx.numel() if S is None else int(S)


def sgmv_shrink(v, x, A, seg_ptr, idx, perm=None, seg_ptr_host=None, S=None):
    """v[p] = x[row(p)] @ A[idx[s]] (fp32), in place; returns v."""
    T, H1 = x.shape
    L, _, r = A.shape
    sph = _host_i32(seg_ptr_host)
    _check(load_library().sgmv_shrink(
        _ptr(v), _ptr(x), _ptr(A), _DTYPES[x.dtype], _ptr(_meta(perm, "perm")),
        _ptr(_meta(seg_ptr, "seg_ptr")), _ptr(_meta(idx, "idx")), _nseg(idx, S), _ptr(sph),
        T, L, H1, r, _stream(x.device)), "sgmv_shrink")
    return v


def sgmv_expand(y, v, B, seg_ptr, idx, scale=1.0, perm=None, seg_ptr_host=None, S=None):
    """y[row(p)] += scale * v[p] @ B[idx[s]], in place; returns y."""
    T, H2 = y.shape
    L, r, _ = B.shape
    sph = _host_i32(seg_ptr_host)
    _check(load_library().sgmv_expand(
        _ptr(y), _DTYPES[y.dtype], _ptr(v), _ptr(B), _DTYPES[B.dtype], float(scale),
        _ptr(_meta(perm, "perm")), _ptr(_meta(seg_ptr, "seg_ptr")), _ptr(_meta(idx, "idx")),
        _nseg(idx, S), _ptr(sph), T, L, H2, r, _stream(y.device)), "sgmv_expand")
    return y


def sgmv_apply(y, x, A, B, seg_ptr, idx, scale=1.0, perm=None, seg_ptr_host=None,
               workspace=None, S=None):
    """y[row(p)] += scale * (x[row(p)] @ A[idx[s]]) @ B[idx[s]], in place; returns y."""
    T, H1 = x.shape
    L, _, r = A.shape
    H2 = y.shape[1]
    sph = _host_i32(seg_ptr_host)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().sgmv_apply(
        _ptr(y), _DTYPES[y.dtype], _ptr(x), _ptr(A), _ptr(B), _DTYPES[x.dtype], float(scale),
        _ptr(_meta(perm, "perm")), _ptr(_meta(seg_ptr, "seg_ptr")), _ptr(_meta(idx, "idx")),
        _nseg(idx, S), _ptr(sph), T, L, H1, H2, r, _ptr(workspace), ws_bytes,
        _stream(x.device)), "sgmv_apply")
    return y


def sgmv_apply_multi(ys, xs, As, Bs, seg_ptr, idx, scale=1.0, perm=None, seg_ptr_host=None,
                     S=None):
    """sgmv_apply for up to 4 problems with the same rows, segments and
    shapes (e.g. a layer's q / k / v): ys[k][row(p)] += scale * (xs[k][row(p)]
    @ As[k][idx[s]]) @ Bs[k][idx[s]], in place, in one launch when the kernel
    allows (the same bits as separate calls); returns ys."""
    P = len(ys)
    if not (len(xs) == len(As) == len(Bs) == P) or P < 1:
        raise ValueError("ys, xs, As and Bs must hold the same number (>= 1) of tensors")
    x0, y0 = xs[0], ys[0]
    T, H1 = x0.shape
    L, _, r = As[0].shape
    H2 = y0.shape[1]
    xshape, ashape, bshape, yshape = (T, H1), (L, H1, r), (L, r, H2), (T, H2)
    tin, ty = x0.dtype, y0.dtype
    for y, x, A, B in zip(ys, xs, As, Bs):
        if x.shape != xshape or A.shape != ashape or B.shape != bshape or y.shape != yshape:
            raise ValueError("the problems' shapes differ")
        if x.dtype != tin or A.dtype != tin or B.dtype != tin or y.dtype != ty:
            raise TypeError("the problems' types differ")
    arr = _PTR_ARRAYS[P] if P < len(_PTR_ARRAYS) else ctypes.c_void_p * P
    _check(load_library().sgmv_apply_multi(
        P, arr(*[t.data_ptr() for t in ys]), _DTYPES[ty], arr(*[t.data_ptr() for t in xs]),
        arr(*[t.data_ptr() for t in As]), arr(*[t.data_ptr() for t in Bs]), _DTYPES[tin],
        float(scale), _ptr(_meta(perm, "perm")), _ptr(_meta(seg_ptr, "seg_ptr")),
        _ptr(_meta(idx, "idx")), _nseg(idx, S), _ptr(_host_i32(seg_ptr_host)), T, L, H1, H2, r,
        _stream(x0.device)), "sgmv_apply_multi")
    return ys


def sgmv_apply_rows(y, x, A, B, row_adapter, scale=1.0, out=None, workspace=None):
    """Group the rows by adapter and apply SGMV in one call; returns y.

    ``out`` = (perm, seg_ptr, idx, S) device int32 tensors (as returned by
    sgmv_build_segments_device) to receive the grouping, or None.
    """
    T, H1 = x.shape
    L, _, r = A.shape
    H2 = y.shape[1]
    ra = _meta(row_adapter, "row_adapter")
    perm = seg_ptr = idx = S = None
    if out is not None:
        perm, seg_ptr, idx, S = (_meta(t, "out") for t in out)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().sgmv_apply_rows(
        _ptr(y), _DTYPES[y.dtype], _ptr(x), _ptr(A), _ptr(B), _DTYPES[x.dtype], float(scale),
        _ptr(ra), T, L, H1, H2, r, _ptr(perm), _ptr(seg_ptr), _ptr(idx), _ptr(S),
        _ptr(workspace), ws_bytes, _stream(x.device)), "sgmv_apply_rows")
    return y


def sgmv_apply_noalloc(y, x, A, B, seg_ptr, idx, scale=1.0, perm=None, seg_ptr_host=None, S=None):
    """sgmv_apply without a caller-provided workspace: for callers that may not
    allocate device memory, the tensor-core path uses a fixed 4 MiB scratch
    array inside the library (see include/sgmv.h).  Calls that overlap on the
    GPU share that array and race; returns y."""
    T, H1 = x.shape
    L, _, r = A.shape
    H2 = y.shape[1]
    sph = _host_i32(seg_ptr_host)
    _check(load_library().sgmv_apply_noalloc(
        _ptr(y), _DTYPES[y.dtype], _ptr(x), _ptr(A), _ptr(B), _DTYPES[x.dtype], float(scale),
        _ptr(_meta(perm, "perm")), _ptr(_meta(seg_ptr, "seg_ptr")), _ptr(_meta(idx, "idx")),
        _nseg(idx, S), _ptr(sph), T, L, H1, H2, r, _stream(x.device)), "sgmv_apply_noalloc")
    return y


def sgmv_fused_workspace_bytes(T: int, H2: int, r: int) -> int:
    return int(load_library().sgmv_fused_workspace_bytes(T, H2, r))


def sgmv_fused_linear_lora(y, x, W, A, B, seg_ptr, idx, scale=1.0, perm=None, S=None,
                           workspace=None):
    """y = x @ W + scale * SGMV delta (the LoRA layer in one pass), written
    into y; returns y.  ``workspace`` (uint8 device tensor of at least
    sgmv_fused_workspace_bytes(T, H2, r) bytes) holds v, its tiles and the
    partial sums; one is allocated when None."""
    T, H1 = x.shape
    L, _, r = A.shape
    H2 = y.shape[1]
    if tuple(W.shape) != (H1, H2):
        raise ValueError("W must be [H1, H2]")
    if W.dtype != x.dtype:
        raise TypeError("W and x types differ")
    nseg = _nseg(idx, S) if idx is not None else 0
    if workspace is None and T > 0:
        workspace = torch.empty(sgmv_fused_workspace_bytes(T, H2, r), dtype=torch.uint8,
                                device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().sgmv_fused_linear_lora(
        _ptr(y), _DTYPES[y.dtype], _ptr(x), _ptr(W), _ptr(A), _ptr(B), _DTYPES[x.dtype],
        float(scale), _ptr(_meta(perm, "perm")), _ptr(_meta(seg_ptr, "seg_ptr")),
        _ptr(_meta(idx, "idx")), nseg, T, L, H1, H2, r, _ptr(workspace), ws_bytes,
        _stream(x.device)), "sgmv_fused_linear_lora")
    return y


def sgmv_load_adapter(A_pool, B_pool, slot, A_src, B_src, stream=None):
    """Copy one adapter (A_src [H1, r], B_src [r, H2]; host -- ideally pinned --
    or device tensors) into slot `slot` of the pools A_pool [L, H1, r] and
    B_pool [L, r, H2], asynchronously on `stream` (default: the current
    stream of the pools' device)."""
    L, H1, r = A_pool.shape
    H2 = B_pool.shape[2]
    if tuple(A_src.shape) != (H1, r) or tuple(B_src.shape) != (r, H2):
        raise ValueError("adapter shapes do not match the pools")
    if A_src.dtype != A_pool.dtype or B_src.dtype != B_pool.dtype or A_pool.dtype != B_pool.dtype:
        raise TypeError("adapter and pool types differ")
    for t in (A_pool, B_pool, A_src, B_src):
        if not t.is_contiguous():
            raise TypeError("tensors must be contiguous")
    st = (stream if stream is not None else torch.cuda.current_stream(A_pool.device)).cuda_stream
    _check(load_library().sgmv_load_adapter(
        _ptr(A_pool), _ptr(B_pool), _DTYPES[A_pool.dtype], int(slot), _ptr(A_src), _ptr(B_src),
        L, H1, H2, r, st), "sgmv_load_adapter")


GATHER_MAX_COPIES = 512


def sgmv_copy_gather(dsts, srcs, stream=None, max_ctas=0):
    """Copy every srcs[i] into dsts[i] (contiguous tensors of equal byte size;
    host -- ideally page-locked -- or device) on `stream` (default: the
    current stream of the current device): one kernel launch for the pairs
    the device reads directly, one copy-engine transfer for each other pair.
    More than GATHER_MAX_COPIES pairs are issued in groups."""
    if len(dsts) != len(srcs):
        raise ValueError("dsts and srcs differ in length")
    for d, s in zip(dsts, srcs):
        if not d.is_contiguous() or not s.is_contiguous():
            raise TypeError("tensors must be contiguous")
        if d.nbytes != s.nbytes:
            raise ValueError("a destination and its source differ in size")
    st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
    lib = load_library()
    for g0 in range(0, len(dsts), GATHER_MAX_COPIES):
        part = range(g0, min(len(dsts), g0 + GATHER_MAX_COPIES))
        n = len(part)
        d = (ctypes.c_void_p * n)(*[dsts[i].data_ptr() for i in part])
        s = (ctypes.c_void_p * n)(*[srcs[i].data_ptr() for i in part])
        b = (ctypes.c_uint64 * n)(*[srcs[i].nbytes for i in part])
        _check(lib.sgmv_copy_gather(n, d, s, b, int(max_ctas), st), "sgmv_copy_gather")


def sgmv_read_floor(src, nbytes, T, L, H1, H2, r, in_dtype=torch.float16, y_dtype=None):
    """Read ``nbytes`` of the device tensor ``src`` with the streaming kernel's
    launch shape for a T-row batch (see include/sgmv.h); returns
    (ctas, cluster) of the grid it launched."""
    y_dtype = in_dtype if y_dtype is None else y_dtype
    if nbytes > src.numel() * src.element_size():
        raise ValueError("nbytes beyond the source tensor")
    ctas, cl = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load_library().sgmv_read_floor(
        _ptr(src), int(nbytes), T, L, H1, H2, r, _DTYPES[in_dtype], _DTYPES[y_dtype],
        ctypes.byref(ctas), ctypes.byref(cl), _stream(src.device)), "sgmv_read_floor")
    return ctas.value, cl.value


def sgmv_debug_inject_wait_timeout(enable: bool) -> None:
    """Make this thread's streaming-kernel launches take the timeout path at
    their first wait (tests of device-side timeout reporting)."""
    _check(load_library().sgmv_debug_inject_wait_timeout(1 if enable else 0),
           "sgmv_debug_inject_wait_timeout")


def sgmv_get_device_error(device=None) -> int:
    """Synchronise the current stream, read and clear the device error word."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    return int(load_library().sgmv_get_device_error(_stream(dev)))
