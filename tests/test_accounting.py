"""Closed forms printed on "Multi-LoRA Serving" (numpy listing output) pin the
roofline accounting (no GPU)."""
import json
import os

import numpy as np

from segmented_gathered_rank_gb300 import accounting as A

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_example.json")


def test_flop_overhead_matches_page():
    g = json.load(open(GOLDEN))
    # "adapter FLOPs overhead vs base matmul: 1.56% (2r/d = 1.56%)" at d=2048, r=16
    assert round(100 * A.flop_overhead_ratio(16, 2048), 2) == g["flop_overhead_percent"]
    assert A.flop_overhead_ratio(16, 2048) == 2 * 16 / 2048


def test_adapter_memory_matches_page():
    g = json.load(open(GOLDEN))
    # "one adapter, one 2048x2048 layer: 0.13 MB vs base layer 8.4 MB" (fp16)
    assert round(A.adapter_bytes(16, 2048, 2048, 2) / 1e6, 2) == g["adapter_layer_mb"]
    assert round(2048 * 2048 * 2 / 1e6, 1) == g["base_layer_mb"]


def test_paging_uses_2r_pages_without_padding():
    # S-LoRA slide 8: rank R -> R pages (per matrix of A and of B)
    assert A.pool_pages([8, 16, 64]) == 2 * (8 + 16 + 64)


def test_bgmv_bytes_counts_distinct_adapters_once():
    ranks = np.full(32, 16)
    ids = np.array([0, 0, 1, 1, 1, -1], np.int32)
    b = A.bgmv_bytes(ids, ranks, 4096, 4096, 2)
    assert b == 2 * 16 * 8192 * 2 + 6 * 4096 * 2 + 2 * 6 * 4096 * 2


def test_layer_flops():
    ranks = np.array([16, 128])
    ids = np.array([0, 1, 1, -1])
    assert A.layer_flops(ids, ranks, 64, 32) == 2 * 4 * 64 * 32 + 2 * (16 * 1 + 128 * 2) * (64 + 32)
