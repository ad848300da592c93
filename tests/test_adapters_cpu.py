"""Slot management of the on-demand adapter pool (host logic, no GPU)."""
import pytest
import torch

from rank_gemv_gb300.adapters import AdapterPool, AdapterPoolFull


def make_pool(L=3):
    pools = [(torch.zeros(L, 8, 4), torch.zeros(L, 4, 16))]
    calls = []

    def loader(slot, weights):
        calls.append((slot, weights))

    pool = AdapterPool(pools, source=lambda n: n, loader=loader, gpu=False)
    return pool, calls


def test_first_use_fills_free_slots_in_order():
    pool, calls = make_pool()
    assert pool.slots_for(["a", "b", "a", "c"]) == [0, 1, 0, 2]
    assert [c[1] for c in calls] == ["a", "b", "c"]  # each adapter loaded once
    assert pool.loads == 3


def test_resident_adapters_are_not_reloaded():
    pool, calls = make_pool()
    pool.slots_for(["a", "b"])
    calls.clear()
    assert pool.slots_for(["b", "a", "b"]) == [1, 0, 1]
    assert calls == []


def test_least_recently_used_is_evicted_first():
    pool, calls = make_pool()
    pool.slots_for(["a", "b", "c"])   # slots 0, 1, 2; recency a < b < c
    pool.slots_for(["a"])             # recency b < c < a
    calls.clear()
    assert pool.slots_for(["d"]) == [1]  # b was least recent
    assert calls == [(1, "d")]
    assert "b" not in pool.resident


def test_adapters_of_the_batch_are_never_evicted():
    pool, calls = make_pool()
    pool.slots_for(["a", "b", "c"])
    calls.clear()
    # a is the least recent, but the batch needs it: b goes
    slots = pool.slots_for(["a", "d"])
    assert slots[0] == 0 and slots[1] == 1
    assert calls == [(1, "d")]


def test_too_many_distinct_adapters_for_the_slots():
    pool, _ = make_pool(L=2)
    with pytest.raises(AdapterPoolFull):
        pool.slots_for(["a", "b", "c"])


def test_evict_frees_the_slot():
    pool, calls = make_pool(L=2)
    pool.slots_for(["a", "b"])
    pool.evict("a")
    calls.clear()
    assert pool.slots_for(["c"]) == [0]
    assert calls == [(0, "c")]


def test_pools_must_share_the_slot_count():
    with pytest.raises(ValueError):
        AdapterPool([(torch.zeros(3, 8, 4), torch.zeros(3, 4, 16)),
                     (torch.zeros(2, 8, 4), torch.zeros(2, 4, 16))], source=lambda n: n,
                    loader=lambda s, w: None, gpu=False)
