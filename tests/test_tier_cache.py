"""Two-tier adapter cache: the oracle pinned to the page's printed table and
to brute force, and the library's native cache against the oracle (host code,
no GPU).

Source: "Multi-LoRA Serving - S-LoRA/Punica Batching, Adapter Hot-Swap &
Memory", section "Memory: slots, tiers and paging" (the adapter-cache
simulation and its printed output, kept in tests/golden/tier_cache_table.json).
"""
import json
import os

import numpy as np
import pytest

from oracle import cache_sim as C
from segmented_gathered_rank_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tier_cache_table.json")


@pytest.fixture(scope="module")
def table():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def trace():
    return I.adapter_request_trace()


def _row_matches(row, g, h, d, n, host_ms, disk_ms):
    return (d == row["disk_loads"] and g + h + d == n
            and f"{100 * g / n:.1f}" == row["gpu_hit_pct"]
            and f"{100 * h / n:.1f}" == row["host_hit_pct"]
            and f"{C.mean_wait_ms(h, d, n, host_ms, disk_ms):.2f}" == row["mean_wait_ms"])


def test_trace_recipe():
    tr = I.adapter_request_trace()
    assert tr.shape == (50000,) and tr.min() >= 0 and tr.max() <= 499
    # the hottest id dominates and every id is drawn at least once
    counts = np.bincount(tr, minlength=500)
    assert counts.argmax() == 0 and (counts > 0).all()
    # LCG from its definition: the first three states from seed 11
    s, us = 11, []
    for _ in range(3):
        s = (1664525 * s + 1013904223) % 2 ** 32
        us.append(s / 2 ** 32)
    assert np.array_equal(I.lcg_uniforms(11, 3), np.array(us))


def test_oracle_reproduces_printed_table(table, trace):
    n = table["requests"]
    for row in table["rows"]:
        g, h, d = C.simulate(trace, row["gpu_slots"], row["host_slots"])
        assert _row_matches(row, g, h, d, n, table["host_ms"], table["disk_ms"]), (row, g, h, d)


def _brute(trace, gpu_slots, host_slots):
    """Recency lists as plain Python lists (oldest first)."""
    gpu, host = [], []
    out = [0, 0, 0]
    for a in trace:
        a = int(a)
        if a in gpu:
            gpu.remove(a)
            gpu.append(a)
            out[0] += 1
            continue
        gpu.append(a)
        if len(gpu) > gpu_slots:
            gpu.pop(0)
        if a in host:
            host.remove(a)
            host.append(a)
            out[1] += 1
        else:
            host.append(a)
            if len(host) > host_slots:
                host.pop(0)
            out[2] += 1
    return tuple(out)


@pytest.mark.parametrize("slots", [(0, 0), (0, 3), (1, 1), (2, 5), (4, 2), (7, 30)])
def test_oracle_against_brute_force(slots):
    rng = np.random.default_rng(5)
    for _ in range(5):
        tr = rng.integers(0, 12, 400)
        assert C.simulate(tr, *slots) == _brute(tr, *slots)


def test_planted_mistakes_break_the_table(table, trace):
    """Plausible slips in a two-tier LRU each miss the printed table."""

    def host_on_every_request(tr, gs, hs):
        gpu, host = C.LruTier(gs), C.LruTier(hs)
        g = h = d = 0
        for a in tr:
            hit_h = host.ask(int(a))
            if gpu.ask(int(a)):
                g += 1
            elif hit_h:
                h += 1
            else:
                d += 1
        return g, h, d

    def fifo(tr, gs, hs):
        class Fifo(C.LruTier):
            def ask(self, key):
                if key in self.keys:
                    return True
                self.keys[key] = None
                if len(self.keys) > self.slots:
                    self.keys.popitem(last=False)
                return False
        gpu, host = Fifo(gs), Fifo(hs)
        g = h = d = 0
        for a in tr:
            if gpu.ask(int(a)):
                g += 1
            elif host.ask(int(a)):
                h += 1
            else:
                d += 1
        return g, h, d

    def off_by_one_capacity(tr, gs, hs):
        return C.simulate(tr, gs + 1, hs)

    n = table["requests"]
    for mutant in (host_on_every_request, fifo, off_by_one_capacity):
        ok = all(_row_matches(r, *mutant(trace, r["gpu_slots"], r["host_slots"]), n, table["host_ms"],
                              table["disk_ms"]) for r in table["rows"])
        assert not ok, mutant.__name__


# ---------------------------------------------------------------------------
# The library's native cache (host code in the C-ABI library)
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def L():
    from segmented_gathered_rank_gb300 import build
    build.build()
    from segmented_gathered_rank_gb300 import lora
    return lora


def test_library_matches_the_oracle_on_the_page_workload(L, table, trace):
    for row in table["rows"]:
        got = L.lora_tier_sim(trace, 500, row["gpu_slots"], row["host_slots"])
        assert got == C.simulate(trace, row["gpu_slots"], row["host_slots"])
        assert _row_matches(row, *got, table["requests"], table["host_ms"], table["disk_ms"])


@pytest.mark.parametrize("slots", [(0, 0), (1, 0), (3, 7), (16, 64), (100, 400)])
def test_library_matches_the_oracle_on_random_traces(L, slots):
    rng = np.random.default_rng(7)
    tr = I.bounded_zipf(rng, 300, 1.05, 20000)
    assert L.lora_tier_sim(tr, 300, *slots) == C.simulate(tr, *slots)


def test_library_touch_reports_tier_and_eviction(L):
    rng = np.random.default_rng(9)
    tr = rng.integers(0, 10, 300)
    c = L.lora_tier_cache_create(10, 3, 5)
    try:
        gpu, host = [], []
        for a in tr.tolist():
            tier, ev = L.lora_tier_cache_touch(c, a)
            # brute-force expectation
            if a in gpu:
                gpu.remove(a)
                gpu.append(a)
                want, want_ev = L.LORA_TIER_GPU, -1
            else:
                gpu.append(a)
                want_ev = gpu.pop(0) if len(gpu) > 3 else -1
                if a in host:
                    host.remove(a)
                    host.append(a)
                    want = L.LORA_TIER_HOST
                else:
                    host.append(a)
                    if len(host) > 5:
                        host.pop(0)
                    want = L.LORA_TIER_DISK
            assert (tier, ev) == (want, want_ev)
            for k in range(10):
                assert L.lora_tier_cache_resident(c, k) == (1 if k in gpu else 0) | (2 if k in host else 0)
    finally:
        L.lora_tier_cache_destroy(c)


def test_library_rejects_bad_arguments(L):
    import ctypes
    counts = (ctypes.c_longlong * 3)()
    tr = np.array([0, 1, 5], np.int32)
    assert L._lib.lora_tier_sim(ctypes.c_void_p(tr.ctypes.data), 3, 5, 1, 1, counts) == L.LORA_ERR_ARG
    assert L._lib.lora_tier_sim(None, 3, 5, 1, 1, counts) == L.LORA_ERR_ARG
    assert L._lib.lora_tier_sim(None, 0, 5, 1, 1, counts) == L.LORA_OK
    h = ctypes.c_void_p()
    assert L._lib.lora_tier_cache_create(ctypes.byref(h), 0, 1, 1) == L.LORA_ERR_ARG
    assert L._lib.lora_tier_cache_create(ctypes.byref(h), 4, -1, 1) == L.LORA_ERR_ARG
    c = L.lora_tier_cache_create(4, 1, 1)
    try:
        with pytest.raises(L.LoraError):
            L.lora_tier_cache_touch(c, 4)
        with pytest.raises(L.LoraError):
            L.lora_tier_cache_resident(c, -1)
    finally:
        L.lora_tier_cache_destroy(c)
