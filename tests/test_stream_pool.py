"""The streamed expert pool's slot map, on the CPU (planning mode: slots are assigned
and counted, nothing is copied), against an independent least-recently-used model."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_topk_gb300 as moe


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()


def _plan(E, slots, H=256, I=128):
    host = torch.zeros(E * moe.moe_pool_record_bytes(H, I), dtype=torch.uint8)
    return moe.StreamPool(host, E, H, I, slots, plan_only=True)


def test_lru_sequence_by_hand():
    sp = _plan(10, 3)
    assert sp.slots == 3 and sp.cache is None
    assert list(sp.map([1, 2])) == [0, 1]            # two misses into empty slots
    assert list(sp.map([2, 3])) == [1, 2]            # hit; miss into the last empty slot
    assert list(sp.map([4])) == [0]                  # evicts 1 (least recently used)
    assert list(sp.map([1, 4, 1])) == [1, 0, 1]      # hit 4; 1 evicts 2 (slot 1); repeats share
    hits, misses, nbytes = sp.stats()
    assert (hits, misses) == (2, 5)
    assert nbytes == 5 * moe.moe_pool_record_bytes(256, 128)


def test_invalid_indices_and_capacity():
    sp = _plan(10, 3)
    assert list(sp.map([7, -1, 12, 7])) == [0, -1, -1, 0]
    with pytest.raises(moe.MoeError) as e:
        sp.map([1, 2, 3, 4])                         # four distinct experts, three slots
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED_SHAPE


class _Lru:
    """Reference model: slots hold experts; a call's experts are resident afterwards; a
    missing expert takes the least recently used slot the call does not use, the lowest
    slot index among equals (never-used slots count as used at time 0)."""

    def __init__(self, C):
        self.slot = {}
        self.owner = [None] * C
        self.last = [0] * C
        self.t = 0
        self.hits = self.misses = 0

    def map(self, idx):
        self.t += 1
        for e in dict.fromkeys(idx):
            if e in self.slot:
                self.last[self.slot[e]] = self.t
                self.hits += 1
        out = []
        for e in idx:
            if e not in self.slot:
                free = [c for c in range(len(self.owner)) if self.last[c] != self.t]
                v = min(free, key=lambda c: (self.last[c], c))
                if self.owner[v] is not None:
                    del self.slot[self.owner[v]]
                self.owner[v], self.slot[e], self.last[v] = e, v, self.t
                self.misses += 1
            out.append(self.slot[e])
        return out


def test_matches_reference_lru_on_zipf_requests():
    rng = np.random.default_rng(3)
    E, C, k = 96, 24, 8
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    sp, ref = _plan(E, C), _Lru(C)
    for _ in range(400):
        idx = rng.choice(E, size=k, replace=False, p=p).astype(np.int32)
        got = sp.map(idx)
        assert list(got) == ref.map([int(v) for v in idx])
        assert len(set(got)) == k                    # distinct experts, distinct slots
    assert sp.stats()[:2] == (ref.hits, ref.misses)
    assert ref.hits > ref.misses                     # the skew makes the cache useful


def test_host_alloc_argument_checks():
    """moe_host_alloc / moe_host_free reject bad arguments before any CUDA call (so this
    runs without a GPU): a null out pointer or zero bytes is MOE_ERR_INVALID_ARG, and
    freeing a null pointer is a no-op."""
    import ctypes
    L = moe.lib()
    p = ctypes.c_void_p()
    node = ctypes.c_int(7)
    assert L.moe_host_alloc(0, 0, ctypes.byref(p), ctypes.byref(node)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_host_alloc(0, 4096, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_host_free(None, 4096) == moe.MOE_OK
