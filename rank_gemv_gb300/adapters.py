"""On-demand adapter loading into the stacked pools.

The pages' serving system keeps only the adapters that requests need resident
and loads the others on demand, in milliseconds ("Punica: Multi-Tenant LoRA
Serving", nubint.ai review, "Proposed method" and findings).  Here a model's
projections each have a stacked pool A [L, H1, r], B [L, r, H2] on the device;
an AdapterPool maps adapter names to the L slots, least recently used first
out, and loads a missing adapter's weights into every projection's pool on a
copy stream: all of its pieces in one sgmv_copy_gather call (one kernel that
reads page-locked host memory directly), or, with gather=False, two
sgmv_load_adapter copy-engine transfers per projection.

Ordering on the GPU:
  * before a slot is overwritten, the copy stream waits for the work already
    queued on the compute stream (SGMV calls may still read the old adapter);
  * after the loads of a batch, the compute stream waits for the copy stream,
    so the batch's SGMV calls see the new weights.
With page-locked host weights the copies overlap with the compute stream's
kernels.

Host logic only: every byte moves through sgmv_copy_gather or
sgmv_load_adapter.
"""
from __future__ import annotations

from collections import OrderedDict
from typing import Callable, Sequence


class AdapterPoolFull(RuntimeError):
    """A batch needs more distinct adapters than the pools have slots."""


class AdapterPool:
    """Resident adapters of a model's projection pools.

    pools:  one (A_pool [L, H1, r], B_pool [L, r, H2]) pair of device tensors
            per projection, all with the same number of slots L.
    source: source(name) -> one (A [H1, r], B [r, H2]) pair per projection,
            host tensors (page-locked for overlap) or device tensors.
    loader: loader(slot, weights) copies one adapter into every pool; the
            default issues sgmv_copy_gather (gather=True) or sgmv_load_adapter
            (gather=False) on the copy stream.
    gather_ctas: CTA cap of the gather kernel (0: four per SM).  64 CTAs
            already read page-locked host memory as fast as the CPU-GPU link
            delivers it (as fast as one large copy-engine transfer) and leave
            the other SMs to the SGMV calls running meanwhile.
    gpu:    False skips all stream handling (host-only use and tests).
    """

    def __init__(self, pools: Sequence, source: Callable, loader: Callable | None = None,
                 copy_stream=None, gpu: bool = True, gather: bool = True, gather_ctas: int = 64):
        self.pools = list(pools)
        if not self.pools:
            raise ValueError("no pools")
        self.L = int(self.pools[0][0].shape[0])
        for A, B in self.pools:
            if A.shape[0] != self.L or B.shape[0] != self.L:
                raise ValueError("pools with different slot counts")
        self.source = source
        self.gpu = gpu
        self.copy_stream = copy_stream
        if gpu and copy_stream is None:
            import torch

            self.copy_stream = torch.cuda.Stream(self.pools[0][0].device)
        self.gather = gather
        self.gather_ctas = gather_ctas
        self.loader = loader if loader is not None else self._load
        self.resident: "OrderedDict[str, int]" = OrderedDict()  # least recent first
        self.free = list(range(self.L))
        self.loads = 0

    def _load(self, slot: int, weights) -> None:
        from . import sgmv

        if not self.gather:
            for (A_pool, B_pool), (A, B) in zip(self.pools, weights):
                sgmv.sgmv_load_adapter(A_pool, B_pool, slot, A, B, stream=self.copy_stream)
            return
        dsts, srcs = [], []
        for (A_pool, B_pool), (A, B) in zip(self.pools, weights):
            for pool, w in ((A_pool, A), (B_pool, B)):
                if tuple(w.shape) != tuple(pool.shape[1:]) or w.dtype != pool.dtype:
                    raise ValueError("adapter shapes or types do not match the pools")
                dsts.append(pool[slot])
                srcs.append(w)
        sgmv.sgmv_copy_gather(dsts, srcs, stream=self.copy_stream, max_ctas=self.gather_ctas)

    def slots_for(self, names: Sequence[str]) -> list[int]:
        """Slot of every name in `names` (one per row of a batch), loading the
        adapters that are not resident.  Raises AdapterPoolFull if the batch
        needs more distinct adapters than there are slots."""
        needed = list(OrderedDict.fromkeys(names))
        if len(needed) > self.L:
            raise AdapterPoolFull(f"{len(needed)} distinct adapters, {self.L} slots")
        missing = [n for n in needed if n not in self.resident]
        for n in needed:
            if n in self.resident:
                self.resident.move_to_end(n)
        if missing:
            evicting = len(missing) > len(self.free)
            if self.gpu and evicting:
                import torch

                # SGMV calls already queued may still read the slots reused below
                self.copy_stream.wait_stream(torch.cuda.current_stream(self.pools[0][0].device))
            want = set(needed)
            for n in missing:
                if self.free:
                    slot = self.free.pop(0)
                else:
                    victim = next(v for v in self.resident if v not in want)
                    slot = self.resident.pop(victim)
                self.loader(slot, self.source(n))
                self.loads += 1
                self.resident[n] = slot
            if self.gpu:
                import torch

                torch.cuda.current_stream(self.pools[0][0].device).wait_stream(self.copy_stream)
        return [self.resident[n] for n in names]

    def evict(self, name: str) -> None:
        """Forget a resident adapter (its slot becomes free)."""
        slot = self.resident.pop(name)
        self.free.append(slot)
