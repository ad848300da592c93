"""The C ABI without a GPU: the library loads, exports what include/sgmv.h
declares, groups rows on the host exactly like the oracle, and rejects bad
arguments with the documented status before touching CUDA."""
import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

import oracle
from tests.golden import load

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    from rank_gemv_gb300 import build, sgmv

    build.build()
    return sgmv.load_library()


def declared_functions():
    text = (ROOT / "include" / "sgmv.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sgmv_\w+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    from rank_gemv_gb300 import sgmv

    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
        assert n in sgmv.SIGNATURES, f"binding lacks {n}"
    assert sorted(sgmv.SIGNATURES) == names


def test_package_exposes_every_binding_function(lib):
    import rank_gemv_gb300

    for n in declared_functions():
        if n == "sgmv_last_error_string":
            continue  # folded into SgmvError's message
        assert callable(getattr(rank_gemv_gb300, n)), n


def test_status_strings(lib):
    from rank_gemv_gb300 import sgmv

    for code, name in sgmv.STATUS.items():
        assert sgmv.sgmv_status_string(code) == name
    assert sgmv.sgmv_status_string(99) == "SGMV_ERR_UNKNOWN"


def test_max_segments_and_workspace(lib):
    from rank_gemv_gb300 import sgmv

    assert sgmv.sgmv_max_segments(32, 32) == 32
    assert sgmv.sgmv_max_segments(8, 3) == 4
    assert sgmv.sgmv_max_segments(0, 5) == 0
    assert sgmv.sgmv_workspace_bytes(100, 4096, 4096, 16) >= 100 * 16 * 4
    assert sgmv.sgmv_workspace_bytes(0, 4096, 4096, 16) == 0


def test_host_grouping_golden(lib):
    from rank_gemv_gb300 import sgmv

    d = load("segments_worked_example.txt")
    perm, seg_ptr, idx = sgmv.sgmv_build_segments(d["row_adapter"], d["L"])
    assert np.array_equal(perm.numpy(), d["perm"])
    assert np.array_equal(seg_ptr.numpy(), d["seg_ptr"])
    assert np.array_equal(idx.numpy(), d["idx"])


@pytest.mark.parametrize("T,L", [(0, 1), (1, 1), (7, 3), (64, 128), (1000, 37), (5000, 2)])
def test_host_grouping_matches_oracle(lib, T, L):
    from rank_gemv_gb300 import sgmv

    rng = np.random.default_rng(T * 31 + L)
    ra = rng.integers(-1, L, size=T).astype(np.int32)
    perm, seg_ptr, idx = sgmv.sgmv_build_segments(ra, L)
    o_perm, o_seg, o_idx = oracle.build_segments(ra, L)
    assert np.array_equal(perm.numpy(), o_perm)
    assert np.array_equal(seg_ptr.numpy(), o_seg)
    assert np.array_equal(idx.numpy(), o_idx)


def test_host_grouping_rejects_bad_ids(lib):
    from rank_gemv_gb300 import sgmv

    for bad in ([0, 3], [-2, 0]):
        with pytest.raises(sgmv.SgmvError) as e:
            sgmv.sgmv_build_segments(bad, 3)
        assert e.value.status == 4


# Host validation happens before any CUDA call, so fake device addresses are
# safe here: each case below must be rejected on the host.
A16 = 0x10000          # 16-byte aligned fake device address
MIS = 0x10008          # misaligned fake device address


def _apply(lib, **kw):
    args = dict(y=A16, y_dt=0, x=A16, A=A16, B=A16, in_dt=0, scale=1.0, perm=None,
                seg_ptr=A16, idx=A16, S=1, sph=None, T=4, L=2, H1=64, H2=64, r=16,
                ws=None, wsb=0, stream=None)
    args.update(kw)
    sph = args["sph"]
    if sph is not None:
        sph = np.ascontiguousarray(sph, dtype=np.int32)
        sph_p = sph.ctypes.data
    else:
        sph_p = None
    return lib.sgmv_apply(args["y"], args["y_dt"], args["x"], args["A"], args["B"], args["in_dt"],
                          args["scale"], args["perm"], args["seg_ptr"], args["idx"], args["S"],
                          sph_p, args["T"], args["L"], args["H1"], args["H2"], args["r"],
                          args["ws"], args["wsb"], args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(r=0), 1), (dict(r=129), 2), (dict(T=-1), 1), (dict(L=0), 1), (dict(S=-1), 1),
    (dict(H1=12), 3), (dict(H2=100), 3), (dict(H1=0), 1), (dict(in_dt=2), 1), (dict(y_dt=7), 1),
    (dict(x=MIS), 3), (dict(A=MIS), 3), (dict(B=MIS), 3), (dict(y=MIS), 3),
    (dict(x=None), 1), (dict(seg_ptr=None), 1), (dict(idx=None), 1),
    (dict(sph=[0, 5]), 8), (dict(sph=[3, 2]), 8), (dict(sph=[-1, 2]), 8),
    (dict(ws=A16, wsb=16), 6),
])
def test_apply_rejects_bad_arguments(lib, kw, status):
    assert _apply(lib, **kw) == status


def test_empty_problems_are_no_ops(lib):
    assert _apply(lib, T=0, S=0, x=None, y=None, A=None, B=None) == 0
    assert _apply(lib, S=0, seg_ptr=None, idx=None) == 0


def test_shrink_expand_reject_bad_arguments(lib):
    assert lib.sgmv_shrink(A16, A16, A16, 0, None, A16, A16, 1, None, 4, 2, 20, 16, None) == 3
    assert lib.sgmv_shrink(A16, MIS, A16, 0, None, A16, A16, 1, None, 4, 2, 64, 16, None) == 3
    assert lib.sgmv_shrink(A16, A16, A16, 0, None, A16, A16, 1, None, 4, 2, 64, 200, None) == 2
    assert lib.sgmv_expand(A16, 3, A16, A16, 0, 1.0, None, A16, A16, 1, None, 4, 2, 64, 16,
                           None) == 1
    assert lib.sgmv_expand(MIS, 0, A16, A16, 0, 1.0, None, A16, A16, 1, None, 4, 2, 64, 16,
                           None) == 3
    assert lib.sgmv_build_segments_device(A16, 4, 40000, A16, A16, A16, A16, None) == 2
    assert lib.sgmv_build_segments_device(A16, -1, 4, A16, A16, A16, A16, None) == 1


def test_apply_rows_rejects_bad_arguments(lib):
    def call(**kw):
        a = dict(y=A16, y_dt=0, x=A16, A=A16, B=A16, in_dt=0, ra=A16, T=4, L=2, H1=64, H2=64, r=16,
                 perm=None, seg=None, idx=None, S=None, ws=None, wsb=0)
        a.update(kw)
        return lib.sgmv_apply_rows(a["y"], a["y_dt"], a["x"], a["A"], a["B"], a["in_dt"], 1.0,
                                   a["ra"], a["T"], a["L"], a["H1"], a["H2"], a["r"], a["perm"],
                                   a["seg"], a["idx"], a["S"], a["ws"], a["wsb"], None)
    assert call(r=0) == 1
    assert call(r=129) == 2
    assert call(H1=20) == 3
    assert call(x=MIS) == 3
    assert call(ra=None) == 1
    assert call(perm=A16) == 1          # metadata outputs: all or none
    assert call(ws=A16, wsb=8) == 6
    assert call(y_dt=5) == 1


@pytest.mark.parametrize("kw", [
    dict(slot=-1), dict(slot=2), dict(L=0), dict(H1=0), dict(r=0), dict(in_dt=2),
    dict(A=None), dict(B=None), dict(a=None), dict(b=None),
])
def test_load_adapter_rejects_bad_arguments(lib, kw):
    args = dict(A=A16, B=A16, in_dt=0, slot=0, a=A16, b=A16, L=2, H1=64, H2=64, r=16)
    args.update(kw)
    assert lib.sgmv_load_adapter(args["A"], args["B"], args["in_dt"], args["slot"], args["a"],
                                 args["b"], args["L"], args["H1"], args["H2"], args["r"],
                                 None) == 1


def test_apply_multi_rejects_bad_arguments(lib):
    import ctypes

    vp = ctypes.c_void_p
    four = (vp * 4)(A16, A16, A16, A16)

    def call(P=2, y=four, x=four, A=four, B=four, **kw):
        a = dict(y_dt=0, in_dt=0, T=4, L=2, H1=64, H2=64, r=16)
        a.update(kw)
        return lib.sgmv_apply_multi(P, y, a["y_dt"], x, A, B, a["in_dt"], 1.0, None, A16, A16, 1,
                                    None, a["T"], a["L"], a["H1"], a["H2"], a["r"], None)
    assert call(T=0) == 0               # nothing to do: returns before any CUDA call
    assert call(P=0) == 1
    assert call(P=5) == 1               # at most four problems
    assert call(y=None) == 1
    assert call(B=None) == 1
    assert call(y=(vp * 4)(A16, None, A16, A16)) == 1
    assert call(x=(vp * 4)(A16, MIS, A16, A16)) == 3
    assert call(r=0) == 1
    assert call(H1=20) == 3
    assert call(y_dt=7) == 1


def test_copy_gather_rejects_bad_arguments(lib):
    import ctypes

    def arr(t, vals):
        return (t * max(1, len(vals)))(*vals)

    vp, u64 = ctypes.c_void_p, ctypes.c_uint64
    d, s, b = arr(vp, [A16, A16]), arr(vp, [A16, A16]), arr(u64, [16, 32])
    assert lib.sgmv_copy_gather(0, None, None, None, 0, None) == 0    # nothing to do
    assert lib.sgmv_copy_gather(-1, d, s, b, 0, None) == 1
    assert lib.sgmv_copy_gather(513, d, s, b, 0, None) == 1          # more than 512 copies
    assert lib.sgmv_copy_gather(2, d, s, b, -1, None) == 1
    assert lib.sgmv_copy_gather(2, None, s, b, 0, None) == 1
    assert lib.sgmv_copy_gather(2, d, None, b, 0, None) == 1
    assert lib.sgmv_copy_gather(2, d, s, None, 0, None) == 1
    assert lib.sgmv_copy_gather(2, arr(vp, [A16, None]), s, b, 0, None) == 1
    assert lib.sgmv_copy_gather(2, d, arr(vp, [None, A16]), b, 0, None) == 1


def test_read_floor_rejects_bad_arguments(lib):
    def call(**kw):
        a = dict(src=A16, n=1 << 20, T=32, L=32, H1=4096, H2=4096, r=16, in_dt=0, y_dt=0)
        a.update(kw)
        return lib.sgmv_read_floor(a["src"], a["n"], a["T"], a["L"], a["H1"], a["H2"], a["r"],
                                   a["in_dt"], a["y_dt"], None, None, None)
    assert call(src=None) == 1
    assert call(n=0) == 1
    assert call(T=0) == 1
    assert call(src=MIS) == 3
    assert call(n=(1 << 20) + 8) == 3   # not a whole number of 16-byte pieces
    assert call(H1=20) == 3
    assert call(r=6) == 2               # the streaming kernel takes r % 4 == 0 only
    assert call(r=129) == 2
    assert call(y_dt=9) == 1


def test_timeout_injection_switch(lib):
    assert lib.sgmv_debug_inject_wait_timeout(1) == 0
    assert lib.sgmv_debug_inject_wait_timeout(0) == 0


def test_fused_linear_lora_rejects_bad_arguments(lib):
    def call(**kw):
        a = dict(y=A16, y_dt=0, x=A16, W=A16, A=A16, B=A16, in_dt=0, perm=None, seg=A16,
                 idx=A16, S=1, T=4, L=2, H1=64, H2=64, r=16, ws=A16, wsb=1 << 20)
        a.update(kw)
        return lib.sgmv_fused_linear_lora(a["y"], a["y_dt"], a["x"], a["W"], a["A"], a["B"],
                                          a["in_dt"], 1.0, a["perm"], a["seg"], a["idx"], a["S"],
                                          a["T"], a["L"], a["H1"], a["H2"], a["r"], a["ws"],
                                          a["wsb"], None)
    assert call(T=129) == 2            # decode batches only
    assert call(r=65) == 2
    assert call(r=0) == 1
    assert call(H1=20) == 3
    assert call(H2=12) == 3
    assert call(W=None) == 1
    assert call(W=MIS) == 3
    assert call(y=MIS) == 3
    assert call(in_dt=2) == 1
    assert call(y_dt=4) == 1
    assert call(ws=None, wsb=0) == 6   # v and the partials need the workspace
    assert call(ws=None, wsb=0, S=0) == 6
    assert call(wsb=16) == 6
    assert call(ws=MIS) == 3
    assert call(T=0, x=None, y=None) == 0
    # v [T][r] fp32, the pair table (1 + 2T int32), T pairs' v tiles ([16][64]
    # 16-bit, two of them for r > 32) and the split partials (8 x 128-column
    # tiles x round32(T) x 128 fp32), each part 256-byte rounded
    def part(T, H2):
        return 8 * ((H2 + 127) // 128) * ((T + 31) // 32 * 32) * 128 * 4
    f = lib.sgmv_fused_workspace_bytes
    assert f(128, 4096, 16) == 128 * 16 * 4 + 1280 + 128 * 2048 + part(128, 4096)
    assert f(3, 64, 5) == 256 + 256 + 3 * 2048 + part(3, 64)
    assert f(100, 11008, 32) == 100 * 32 * 4 + 1024 + 100 * 2048 + part(100, 11008)
    assert f(7, 200, 64) == 7 * 64 * 4 + 256 + 7 * 4096 + part(7, 200)
    assert f(0, 4096, 16) == 0


def test_multi_binding_marshals_each_problems_pointers(monkeypatch):
    """The Python side of sgmv_apply_multi: the arrays it hands the C ABI hold
    each problem's data pointers in order, and mismatched problems are
    refused before the library is called."""
    import torch

    from rank_gemv_gb300 import sgmv

    calls = []

    class Recorder:
        def sgmv_apply_multi(self, *args):
            calls.append(args)
            return 0

    monkeypatch.setattr(sgmv, "load_library", lambda: Recorder())
    monkeypatch.setattr(sgmv, "_stream", lambda device: None)
    T, H1, H2, L, r = 6, 32, 48, 3, 8
    P = 3
    xs = [torch.zeros(T, H1, dtype=torch.half) for _ in range(P)]
    As = [torch.zeros(L, H1, r, dtype=torch.half) for _ in range(P)]
    Bs = [torch.zeros(L, r, H2, dtype=torch.half) for _ in range(P)]
    ys = [torch.zeros(T, H2, dtype=torch.float32) for _ in range(P)]
    seg = torch.tensor([0, 2, 6], dtype=torch.int32)
    idx = torch.tensor([2, 0], dtype=torch.int32)
    sgmv.sgmv_apply_multi(ys, xs, As, Bs, seg, idx, 0.5, seg_ptr_host=seg)
    (a,) = calls
    assert a[0] == P
    for arr, ts in ((a[1], ys), (a[3], xs), (a[4], As), (a[5], Bs)):
        assert [arr[k] for k in range(P)] == [t.data_ptr() for t in ts]
    assert a[2] == sgmv.SGMV_F32 and a[6] == sgmv.SGMV_F16
    assert a[7] == 0.5 and a[8] is None and a[9] == seg.data_ptr() and a[10] == idx.data_ptr()
    assert a[11] == 2 and a[13:18] == (T, L, H1, H2, r)
    with pytest.raises(ValueError):
        sgmv.sgmv_apply_multi(ys, xs[:2], As, Bs, seg, idx)
    with pytest.raises(ValueError):
        sgmv.sgmv_apply_multi([], [], [], [], seg, idx)
    with pytest.raises(ValueError):
        sgmv.sgmv_apply_multi(ys, xs[:2] + [torch.zeros(T, H1 + 8, dtype=torch.half)], As, Bs,
                              seg, idx)
    with pytest.raises(TypeError):
        sgmv.sgmv_apply_multi(ys, xs, As[:2] + [As[2].bfloat16()], Bs, seg, idx)
    assert len(calls) == 1


def test_a_missing_library_fails_loudly(tmp_path):
    """No CPU fallback: without the built library every entry point raises."""
    from rank_gemv_gb300 import sgmv

    with pytest.raises(RuntimeError, match="is not built"):
        sgmv.load_library(tmp_path / "libsgmv.so")
