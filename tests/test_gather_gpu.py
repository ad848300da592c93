"""sgmv_copy_gather: many copies in one call, bit for bit.

Every copy the device reads directly (its own memory or page-locked host
memory, 16-byte aligned, a multiple of 16 bytes) goes through the one gather
kernel; every other copy through the copy engine.  Each case checks the
destination bytes against the source, that the bytes around every destination
are untouched, and whether the kernel was launched.
"""
import pytest
import torch

from tests.gpu_helpers import check_error_word

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def rand_bytes(n, seed, pin=False, device=None):
    g = torch.Generator().manual_seed(seed)
    t = torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)
    if device is not None:
        return t.to(device)
    return t.pin_memory() if pin else t


def run(pairs, max_ctas=0):
    """pairs: (dst view, src view); every dst a view of one guarded buffer.
    Returns the launch count."""
    from rank_gemv_gb300 import sgmv

    sgmv.sgmv_copy_gather([d for d, _ in pairs], [s for _, s in pairs], max_ctas=max_ctas)
    n = sgmv.load_library().sgmv_last_launch_count()
    torch.cuda.synchronize()
    check_error_word(0)
    return n


def layout(sizes, align=16, gap=64):
    """Offsets of consecutive pieces in one buffer, `gap` guard bytes apart."""
    offs, o = [], gap
    for n in sizes:
        o = (o + align - 1) // align * align
        offs.append(o)
        o += n + gap
    return offs, o


def check(buf, sentinel, offs, srcs):
    got = buf.cpu()
    mask = torch.ones(got.numel(), dtype=torch.bool)
    for o, s in zip(offs, srcs):
        assert torch.equal(got[o:o + s.numel()], s.cpu()), f"piece at {o}"
        mask[o:o + s.numel()] = False
    assert bool((got[mask] == sentinel).all()), "bytes outside the pieces changed"


SIZES = [16, 48, 512, 496, 528, 4096 + 16, 32768, 352 * 1024, 160, 65536 + 48]


def test_pinned_host_to_device_one_launch():
    from rank_gemv_gb300 import build

    build.build()
    srcs = [rand_bytes(n, 10 + i, pin=True) for i, n in enumerate(SIZES)]
    offs, total = layout(SIZES)
    buf = torch.full((total,), 0xA5, dtype=torch.uint8, device=DEV)
    assert run([(buf[o:o + s.numel()], s) for o, s in zip(offs, srcs)]) == 1
    check(buf, 0xA5, offs, srcs)


def test_device_to_device_and_device_to_pinned_host():
    srcs = [rand_bytes(n, 30 + i, device=DEV) for i, n in enumerate(SIZES)]
    offs, total = layout(SIZES, gap=32)
    buf = torch.full((total,), 0x3C, dtype=torch.uint8, device=DEV)
    assert run([(buf[o:o + s.numel()], s) for o, s in zip(offs, srcs)]) == 1
    check(buf, 0x3C, offs, srcs)
    host = torch.full((total,), 0x5A, dtype=torch.uint8).pin_memory()
    assert run([(host[o:o + s.numel()], s) for o, s in zip(offs, srcs)]) == 1
    check(host, 0x5A, offs, srcs)


def test_pageable_sources_take_the_copy_engine():
    srcs = [rand_bytes(n, 50 + i) for i, n in enumerate(SIZES)]  # not page-locked
    offs, total = layout(SIZES)
    buf = torch.full((total,), 0x11, dtype=torch.uint8, device=DEV)
    assert run([(buf[o:o + s.numel()], s) for o, s in zip(offs, srcs)]) == 0
    check(buf, 0x11, offs, srcs)


def test_unaligned_pieces_mixed_with_aligned_ones():
    # odd sizes and 2-byte-aligned addresses go through the copy engine, the
    # rest through the kernel, all in one call
    sizes = [16, 17, 1000, 512, 30, 4096, 2, 777]
    srcs = []
    for i, n in enumerate(sizes):
        s = rand_bytes(n + 16, 70 + i, pin=True)
        srcs.append(s[2:2 + n] if i % 3 == 1 else s[:n])
    offs, total = layout(sizes, align=2)
    buf = torch.full((total,), 0x77, dtype=torch.uint8, device=DEV)
    assert run([(buf[o:o + s.numel()], s) for o, s in zip(offs, srcs)]) == 1
    check(buf, 0x77, offs, srcs)


def test_one_cta_strides_over_every_chunk():
    sizes = [8 * 1024 * 1024 + 16, 48, 1 << 20]
    srcs = [rand_bytes(n, 90 + i, pin=True) for i, n in enumerate(sizes)]
    offs, total = layout(sizes)
    buf = torch.full((total,), 0x99, dtype=torch.uint8, device=DEV)
    assert run([(buf[o:o + s.numel()], s) for o, s in zip(offs, srcs)], max_ctas=1) == 1
    check(buf, 0x99, offs, srcs)


def test_zero_sized_pieces_and_many_copies():
    from rank_gemv_gb300 import sgmv

    # 600 copies: the binding issues them as 512 + 88
    sizes = [(16 * (1 + (7 * i) % 40)) if i % 50 else 0 for i in range(600)]
    srcs = [rand_bytes(n, 200 + i, pin=True) for i, n in enumerate(sizes)]
    offs, total = layout(sizes)
    buf = torch.full((total,), 0xC3, dtype=torch.uint8, device=DEV)
    run([(buf[o:o + s.numel()], s) for o, s in zip(offs, srcs)])
    check(buf, 0xC3, offs, srcs)
    # a zero-sized copy may have null pointers
    import ctypes

    lib = sgmv.load_library()
    one = rand_bytes(64, 7, pin=True)
    dst = torch.zeros(64, dtype=torch.uint8, device=DEV)
    d = (ctypes.c_void_p * 2)(None, dst.data_ptr())
    s = (ctypes.c_void_p * 2)(None, one.data_ptr())
    b = (ctypes.c_uint64 * 2)(0, 64)
    assert lib.sgmv_copy_gather(2, d, s, b, 0, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), one)


def test_ordered_after_earlier_work_on_the_stream():
    # the source is written by a kernel queued just before the copy
    n = 1 << 22
    src = torch.zeros(n, dtype=torch.uint8, device=DEV)
    dst = torch.zeros(n, dtype=torch.uint8, device=DEV)
    pattern = rand_bytes(n, 3, device=DEV)
    for _ in range(3):
        src.copy_(pattern)
        assert run([(dst, src)]) == 1
        assert torch.equal(dst, pattern)
        pattern = pattern.add_(1)


def test_llama7b_adapter_pieces_into_slot_views():
    # one Llama-2-7B adapter (224 projections x A, B) from page-locked host
    # memory into slot 1 of every projection's pool
    from rank_gemv_gb300 import workloads as wl

    r = 16
    g = torch.Generator().manual_seed(11)
    pools, srcs = [], []
    for layer in range(wl.LLAMA7B_LAYERS):
        for _, H1, H2 in wl.LLAMA7B_PROJ:
            pools.append(torch.zeros(2, H1, r, dtype=torch.half, device=DEV))
            srcs.append(torch.randn(H1, r, generator=g).half().pin_memory())
            pools.append(torch.zeros(2, r, H2, dtype=torch.half, device=DEV))
            srcs.append(torch.randn(r, H2, generator=g).half().pin_memory())
    assert run([(p[1], s) for p, s in zip(pools, srcs)]) == 1
    for p, s in zip(pools, srcs):
        assert torch.equal(p[1].cpu(), s)
        assert not bool(p[0].any())


def test_bad_arguments_are_refused():
    from rank_gemv_gb300 import sgmv

    a = torch.zeros(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError):
        sgmv.sgmv_copy_gather([a], [a[:32]])
    with pytest.raises(sgmv.SgmvError) as e:
        sgmv.sgmv_copy_gather([a], [a], max_ctas=-1)
    assert e.value.status == 1
