"""Host helpers of bench.py that need no GPU.

The end-to-end measurement moves a step's x, y and row -> adapter ids in one
copy: they live in one byte buffer as views at 256-byte-aligned offsets (the
C ABI wants 16-byte-aligned rows).  The views must hold the original values,
not overlap, and together span the buffer.
"""
import torch

import bench


def test_packed_views_hold_the_tensors_without_overlap():
    X = torch.randn(3, 40, dtype=torch.float16)
    Y = torch.randn(3, 24, dtype=torch.float32)
    ra = torch.tensor([2, -1, 0], dtype=torch.int32)
    buf, (x, y, r) = bench._packed([X, Y, ra], "cpu")
    assert torch.equal(x, X) and torch.equal(y, Y) and torch.equal(r, ra)
    base = buf.data_ptr()
    spans = sorted((v.data_ptr() - base, v.data_ptr() - base + v.nbytes) for v in (x, y, r))
    assert all(lo % 256 == 0 for lo, _ in spans)
    assert all(spans[i][1] <= spans[i + 1][0] for i in range(len(spans) - 1))
    assert spans[-1][1] == buf.nbytes
    # writing through the buffer is seen by the views (one copy moves all three)
    buf.zero_()
    assert not x.any() and not y.any() and not r.any()
