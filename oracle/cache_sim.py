"""CPU oracle of the two-tier adapter cache.

TEST INFRASTRUCTURE ONLY: the tests are its only callers; the library never
imports it and it imports nothing from the library.

Follows the adapter-cache simulation of "Multi-LoRA Serving - S-LoRA/Punica
Batching, Adapter Hot-Swap & Memory" (section "Memory: slots, tiers and
paging"), step by step: every request first asks the GPU tier; a GPU tier
that already holds the adapter counts a GPU hit; otherwise the host tier is
asked, counting a host hit or, when it misses too, a disk load.  Asking a
tier makes the adapter its most recently used entry (inserting it if absent)
and, when that leaves the tier over its slot count, drops its least recently
used entry.  The mean load wait per request weighs host hits and disk loads
by their example latencies (3 ms and 120 ms on the page).

Parity status: pinned by the page's printed table (disk loads exactly, hit
rates to 0.1 %, mean wait to 0.01 ms, for four slot configurations) in
``tests/test_tier_cache.py``, and by brute-force recency lists on small
traces there.
"""
from __future__ import annotations

from collections import OrderedDict


class LruTier:
    """One tier: keys in recency order, oldest first."""

    def __init__(self, slots: int):
        self.slots = slots
        self.keys: OrderedDict[int, None] = OrderedDict()

    def ask(self, key: int) -> bool:
        hit = key in self.keys
        if hit:
            del self.keys[key]
        self.keys[key] = None
        if len(self.keys) > self.slots:
            self.keys.popitem(last=False)
        return hit


def simulate(trace, gpu_slots: int, host_slots: int):
    """(GPU hits, host hits, disk loads) over the request trace."""
    gpu, host = LruTier(gpu_slots), LruTier(host_slots)
    g = h = d = 0
    for a in trace:
        a = int(a)
        if gpu.ask(a):
            g += 1
        elif host.ask(a):
            h += 1
        else:
            d += 1
    return g, h, d


def mean_wait_ms(host_hits: int, disk_loads: int, requests: int, host_ms: float = 3.0,
                 disk_ms: float = 120.0) -> float:
    """Mean load wait per request: host hits and disk loads at their latencies."""
    return (host_hits * host_ms + disk_loads * disk_ms) / requests
