"""The seeded input generators (CPU only): shapes, determinism, distributions."""
import torch

from rank_gemv_gb300 import workloads as wl


def test_named_workload_shapes():
    w = wl.make("tiny")
    assert (w.T, w.L, w.H1, w.H2, w.r) == (8, 4, 512, 512, 8)
    assert w.row_adapter.tolist() == [0, 0, 1, 1, 2, 2, 3, 3]
    assert w.X.dtype == torch.float16 and torch.count_nonzero(w.Y0) == 0
    w = wl.make("decode-distinct")
    assert w.row_adapter.tolist() == list(range(32)) and w.A.shape == (32, 4096, 16)
    w = wl.make("decode-shared")
    assert w.row_adapter.tolist() == [0] * 32
    w = wl.make("decode-zipf", seed=3)
    assert w.B.shape == (128, 16, 11008) and w.T == 64
    assert torch.all(w.row_adapter[1:] >= w.row_adapter[:-1])
    w = wl.make("prefill", seed=1)
    lens = torch.bincount(w.row_adapter.long(), minlength=8)
    assert lens.numel() == 8 and int(lens.min()) >= 64 and int(lens.max()) <= 512
    assert w.X.dtype == torch.bfloat16 and w.Y0.dtype == torch.float32 and w.r == 64


def test_seeded_and_reproducible():
    a = wl.make("decode-zipf", seed=5)
    b = wl.make("decode-zipf", seed=5)
    c = wl.make("decode-zipf", seed=6)
    assert torch.equal(a.X, b.X) and torch.equal(a.row_adapter, b.row_adapter)
    assert not torch.equal(a.X, c.X)


def test_distribution_scales():
    w = wl.make("decode-distinct")
    assert abs(w.X.float().std().item() - 1.0) < 0.02
    assert abs(w.A.float().std().item() * 4096 ** 0.5 - 1.0) < 0.02
    assert abs(w.B.float().std().item() * 16 ** 0.5 - 1.0) < 0.02


def test_zipf_is_skewed():
    g = torch.Generator().manual_seed(0)
    ids = wl.zipf_ids(g, 20000, 128)
    counts = torch.bincount(ids.long(), minlength=128).double()
    # p(1)/p(2) = 2^1.5 for a Zipf(1.5) law
    assert abs(counts[0] / counts[1] - 2 ** 1.5) < 0.25
    assert int(ids.min()) >= 0 and int(ids.max()) <= 127


def test_shuffled_rows_keep_the_multiset():
    a = wl.make("prefill", seed=2)
    b = wl.make("prefill", seed=2, shuffle_rows=True)
    assert torch.equal(torch.sort(a.row_adapter).values, torch.sort(b.row_adapter).values)
    assert not torch.equal(a.row_adapter, b.row_adapter)


def test_algorithmic_bytes():
    w = wl.make("decode-distinct")
    # 32 adapters x (4096x16 + 16x4096) fp16 + X + Y read and written
    assert w.bytes_moved() == 32 * 2 * 65536 * 2 + 32 * 4096 * 2 + 2 * 32 * 4096 * 2
    assert wl.make("decode-shared").bytes_moved() == 2 * 65536 * 2 + 32 * 4096 * 2 * 3
