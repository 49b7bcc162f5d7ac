"""The expert store's host policy (qmm_lru, no device): hand cases for each
rule of include/qmm.h, then long random request sequences against a plain
Python model of the same rules (an ordered dict in recency order)."""
import random
from collections import OrderedDict

import pytest


@pytest.fixture(scope="module")
def qmm():
    from block_quantized_int4_gb300 import _build
    _build.build()
    from block_quantized_int4_gb300 import qmm as m
    return m


class RefLru:
    """Model: `res` maps key -> slot, least recent first."""

    def __init__(self, n_keys, n_slots):
        self.n_keys, self.n_slots = n_keys, n_slots
        self.res = OrderedDict()
        self.free = list(range(n_slots))  # slot 0 first
        self.last_use = set()
        self.stats = dict(hits=0, misses=0, evictions=0, prefetched=0)

    def _victim(self, protected):
        if self.free:
            return None, self.free.pop(0)
        for k, s in self.res.items():  # least recent first
            if k not in protected:
                return k, s
        return None, -1

    def request(self, keys, use=True):
        if use and len(set(keys)) > self.n_slots:
            raise ValueError("does not fit")
        protected = set(k for k in keys if k in self.res)
        if use:
            self.stats["hits"] += len(protected)
            self.last_use = set(keys)
            guard = self.last_use
        else:
            guard = self.last_use | protected
        slots, loads = [], []
        for k in keys:
            if k in self.res:
                self.res.move_to_end(k)
                slots.append(self.res[k])
                continue
            old, s = self._victim(guard)
            if s < 0:
                slots.append(-1)
                continue
            if old is not None:
                del self.res[old]
                self.stats["evictions"] += 1
            self.res[k] = s
            self.stats["misses" if use else "prefetched"] += 1
            if not use:
                guard = guard | {k}
            loads.append((k, s))
            slots.append(s)
        return slots, loads


def test_lru_hand_cases(qmm):
    c = qmm.Lru(8, 2)
    assert c.request([0]) == ([0], [(0, 0)])
    assert c.request([1]) == ([1], [(1, 1)])
    assert c.request([2]) == ([0], [(2, 0)])         # evicts key 0, the least recent
    assert c.slot_of(0) == -1 and c.slot_of(2) == 0
    # keys of one request protect each other: 1 is least recent, but is in the request
    assert c.request([3, 1]) == ([0, 1], [(3, 0)])  # evicts key 2 instead
    assert c.stats() == dict(hits=1, misses=4, evictions=2, prefetched=0)
    # a repeated key counts once
    c.request([3, 3, 1, 3])
    assert c.stats()["hits"] == 3
    # prefetch leaves the last use request's keys alone: nothing free, so skipped
    assert c.request([5], use=False) == ([-1], [])
    # more distinct keys than slots: error, nothing changes
    with pytest.raises(qmm.QmmError):
        c.request([4, 5, 6])
    assert c.slot_of(3) == 0 and c.slot_of(1) == 1
    # after a request that uses only key 3, a prefetch may take key 1's slot
    c.request([3])
    assert c.request([6], use=False) == ([1], [(6, 1)])
    assert c.request([6]) == ([1], [])               # prefetched: a hit
    assert c.stats()["prefetched"] == 1


def test_lru_bad_keys(qmm):
    c = qmm.Lru(4, 2)
    with pytest.raises(qmm.QmmError):
        c.request([4])
    with pytest.raises(qmm.QmmError):
        c.request([-1])
    assert c.request([]) == ([], [])


@pytest.mark.parametrize("n_keys,n_slots,seed", [(256, 48, 1), (64, 64, 2), (32, 5, 3), (1000, 200, 4)])
def test_lru_against_model(qmm, n_keys, n_slots, seed):
    rng = random.Random(seed)
    weights = [1.0 / (i + 1) ** 0.8 for i in range(n_keys)]  # skewed popularity
    c, ref = qmm.Lru(n_keys, n_slots), RefLru(n_keys, n_slots)
    for step in range(600):
        use = rng.random() < 0.75
        n = rng.randint(0, min(12, n_slots) if use else 12)
        keys = rng.choices(range(n_keys), weights=weights, k=n)
        if use and len(set(keys)) > n_slots:
            continue
        got = c.request(keys, use=use)
        want = ref.request(keys, use=use)
        assert got == want, (step, keys, use)
        if step % 50 == 0:
            assert all(c.slot_of(k) == ref.res.get(k, -1) for k in range(n_keys))
    assert c.stats() == ref.stats
