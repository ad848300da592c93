"""Seeded synthetic SGMV inputs shaped like multi-LoRA Llama-7B serving.

This module only draws random numbers and lays them out; it holds none of the
SGMV arithmetic.  The tests feed the same tensors to the CUDA path and to the
fp64 oracle, and the benchmark times the CUDA path on them.

The pages' workloads are multi-LoRA serving of a Llama-2-7B base with many
adapters, request distributions uniform or skewed across adapters, adapter
counts from a few to about a hundred and batches of 1 to 128 ("Punica: when
LoRA fine-tuned models need multi-tenant serving", omica.com.cn article,
§4.1).  No dataset is named; these synthetic tensors stand in for it.

Distributions (every workload):
    X ~ N(0, 1), A ~ N(0, 1/H1), B ~ N(0, 1/r)   (variance, so the LoRA delta
    has RMS about |scale|), Y0 = 0 unless a test asks for N(0, 1),
    scale = 1.
Named workloads:
    tiny             T=8, 4 segments of 2 rows, adapters 0..3, H1=H2=512, r=8, fp16
    decode-distinct  T=32, each row its own adapter out of 32, H1=H2=4096, r=16, fp16
    decode-shared    decode-distinct with every row on adapter 0
    decode-zipf      T=64, ids ~ Zipf(1.5) truncated to 128 adapters, rows sorted
                     by id, H1=4096, H2=11008, r=16, fp16
    prefill          8 segments, lengths uniform on the integers 64..512, adapters
                     0..7, H1=4096, H2=11008, r=64, bf16 (Y fp32 by default)
    llama7b-q        one projection of llama7b-stack: T=128 rows on 128 adapters,
                     4096->4096, r=16, fp16 (a small case of the same launch)
    llama7b-stack    32 layers x 7 projections of Llama-2-7B (q,k,v,o 4096->4096,
                     gate,up 4096->11008, down 11008->4096), r=16, T=128 rows,
                     row t on adapter t out of 128, fp16; drawn per projection
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

F16, BF16, F32 = torch.float16, torch.bfloat16, torch.float32


@dataclass
class Workload:
    name: str
    T: int
    L: int
    H1: int
    H2: int
    r: int
    dtype: torch.dtype
    y_dtype: torch.dtype
    scale: float
    row_adapter: torch.Tensor  # int32 [T], adapter id per physical row (-1 = none)
    X: torch.Tensor            # [T, H1]
    A: torch.Tensor            # [L, H1, r]
    B: torch.Tensor            # [L, r, H2]
    Y0: torch.Tensor           # [T, H2]
    meta: dict = field(default_factory=dict)

    def to(self, device) -> "Workload":
        out = Workload(**{**self.__dict__})
        for k in ("X", "A", "B", "Y0"):
            setattr(out, k, getattr(self, k).to(device))
        out.row_adapter = self.row_adapter.clone()
        return out

    def bytes_moved(self, distinct_ids=None) -> int:
        """Algorithmic HBM bytes of one SGMV update: the A and B slices of every
        distinct adapter used, X read once, Y read and written once."""
        ids = torch.unique(self.row_adapter) if distinct_ids is None else distinct_ids
        n = int((ids >= 0).sum())
        es = torch.tensor([], dtype=self.dtype).element_size()
        ys = torch.tensor([], dtype=self.y_dtype).element_size()
        return (n * (self.H1 * self.r + self.r * self.H2) * es
                + self.T * self.H1 * es + 2 * self.T * self.H2 * ys)

    def flops(self) -> int:
        used = int((self.row_adapter >= 0).sum())
        return 2 * used * (self.H1 * self.r + self.r * self.H2)


LLAMA7B_PROJ = [  # (name, H1, H2)
    ("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
    ("gate", 4096, 11008), ("up", 4096, 11008), ("down", 11008, 4096),
]
LLAMA7B_LAYERS = 32


def _normal(g, shape, std, dtype, device="cpu"):
    return (torch.randn(shape, generator=g, dtype=F32, device=device) * std).to(dtype)


def draw(T, L, H1, H2, r, row_adapter, *, dtype=F16, y_dtype=None, seed=0,
         y0="zeros", scale=1.0, name="custom", generator=None, meta=None) -> Workload:
    """Draw X, A, B, Y0 for a given row -> adapter assignment (CPU tensors)."""
    y_dtype = dtype if y_dtype is None else y_dtype
    g = generator if generator is not None else torch.Generator().manual_seed(seed)
    ra = torch.as_tensor(row_adapter, dtype=torch.int32).reshape(-1)
    assert ra.numel() == T
    X = _normal(g, (T, H1), 1.0, dtype)
    A = _normal(g, (L, H1, r), H1 ** -0.5, dtype)
    B = _normal(g, (L, r, H2), r ** -0.5, dtype)
    if y0 == "zeros":
        Y0 = torch.zeros((T, H2), dtype=y_dtype)
    elif y0 == "randn":
        Y0 = _normal(g, (T, H2), 1.0, y_dtype)
    else:
        raise ValueError(y0)
    return Workload(name, T, L, H1, H2, r, dtype, y_dtype, float(scale), ra, X, A, B, Y0,
                    dict(meta or {}))


def zipf_ids(g, n, L, a=1.5):
    """n ids drawn from p(k) ~ k^-a over k = 1..L (truncated Zipf), returned as k-1."""
    k = torch.arange(1, L + 1, dtype=torch.float64)
    p = k.pow(-a)
    p = p / p.sum()
    return torch.multinomial(p, n, replacement=True, generator=g).to(torch.int32)


def make(name: str, seed: int = 0, *, y_dtype=None, y0="zeros", shuffle_rows=False) -> Workload:
    """One of the named workloads (CPU tensors).  ``shuffle_rows`` stores the
    rows in a seeded random order, so that grouping needs a real permutation."""
    g = torch.Generator().manual_seed(seed)
    if name == "tiny":
        T, L, H1, H2, r, dt = 8, 4, 512, 512, 8, F16
        ra = torch.arange(4, dtype=torch.int32).repeat_interleave(2)
    elif name in ("decode-distinct", "decode-shared"):
        T, L, H1, H2, r, dt = 32, 32, 4096, 4096, 16, F16
        ra = (torch.arange(T, dtype=torch.int32) if name == "decode-distinct"
              else torch.zeros(T, dtype=torch.int32))
    elif name == "decode-zipf":
        T, L, H1, H2, r, dt = 64, 128, 4096, 11008, 16, F16
        ra = torch.sort(zipf_ids(g, T, L)).values
    elif name == "llama7b-q":
        # one projection of llama7b-stack (q of layer 0): a small case of the
        # same kernel launch, for profiling
        T, L, H1, H2, r, dt = 128, 128, 4096, 4096, 16, F16
        ra = torch.arange(T, dtype=torch.int32)
    elif name == "prefill":
        L, H1, H2, r, dt = 8, 4096, 11008, 64, BF16
        lens = torch.randint(64, 513, (8,), generator=g, dtype=torch.int64)
        ra = torch.arange(8, dtype=torch.int32).repeat_interleave(lens)
        T = int(lens.sum())
        y_dtype = F32 if y_dtype is None else y_dtype
    else:
        raise ValueError(f"unknown workload {name!r}")
    if shuffle_rows:
        ra = ra[torch.randperm(T, generator=g)]
    return draw(T, L, H1, H2, r, ra, dtype=dt, y_dtype=y_dtype, y0=y0, name=name,
                generator=g, meta={"seed": seed})


def base_weight(H1: int, H2: int, *, dtype=F16, seed: int = 0, device="cpu") -> torch.Tensor:
    """Weight W [H1, H2] of the base linear layer for the fused layer
    y = x W + LoRA delta, W ~ N(0, 1/H1) (variance), so that x W has RMS
    about 1 like the delta."""
    g = torch.Generator(device=device).manual_seed(seed)
    return _normal(g, (H1, H2), H1 ** -0.5, dtype, device)


def stack_seed(seed: int, layer: int, proj: int) -> int:
    return 1000 * seed + 7 * layer + proj


def stack_projection(seed: int, layer: int, proj: int, device="cpu", T=128, L=128, r=16,
                     dtype=F16):
    """(X, A, B, Y0) of one Llama-2-7B projection in the llama7b-stack workload.

    Drawn with a generator on ``device`` seeded from (seed, layer, proj), so a
    projection can be drawn alone, on the GPU for the benchmark or again on the
    same device for a sampled check."""
    _, H1, H2 = LLAMA7B_PROJ[proj]
    g = torch.Generator(device=device).manual_seed(stack_seed(seed, layer, proj))
    X = _normal(g, (T, H1), 1.0, dtype, device)
    A = _normal(g, (L, H1, r), H1 ** -0.5, dtype, device)
    B = _normal(g, (L, r, H2), r ** -0.5, dtype, device)
    Y0 = torch.zeros((T, H2), dtype=dtype, device=device)
    return X, A, B, Y0


def stack_row_adapter(T=128) -> torch.Tensor:
    return torch.arange(T, dtype=torch.int32)
