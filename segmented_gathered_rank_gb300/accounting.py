"""Algorithmic work of one adapted projection: bytes and FLOPs.

These are the figures a roofline is computed from (what the operation must
move or compute at minimum), not what a kernel happens to move.

Closed forms from "Multi-LoRA Serving" (numpy listing and its printed
output): the adapter term of one d x d layer costs 2 * batch * r * d * 2
FLOPs against the base product's 2 * batch * d * d, a ratio of 2r/d; one
adapter on one d x d layer holds 2 * r * d values (A and B).
"""
from __future__ import annotations

import numpy as np


def adapter_flops(tokens_per_rank: dict, h_in: int, h_out: int) -> int:
    """FLOPs of the adapter term: 2 * r * (h_in + h_out) per adapted token.

    ``tokens_per_rank`` maps rank -> number of tokens using an adapter of that rank.
    """
    return int(sum(2 * r * (h_in + h_out) * n for r, n in tokens_per_rank.items()))


def base_flops(T: int, h_in: int, h_out: int) -> int:
    return 2 * T * h_in * h_out


def flop_overhead_ratio(r: int, d: int) -> float:
    """Adapter FLOPs / base FLOPs for a d x d layer at rank r (= 2r/d)."""
    return adapter_flops({r: 1}, d, d) / base_flops(1, d, d)


def adapter_bytes(r: int, h_in: int, h_out: int, esize: int) -> int:
    """Bytes of one adapter (A and B) on one projection."""
    return r * (h_in + h_out) * esize


def pool_pages(ranks) -> int:
    """Pages a set of adapters occupies on one matrix: 2r each, no padding."""
    return int(2 * np.sum(np.asarray(ranks, np.int64)))


def tokens_per_rank(token_adapter, ranks) -> dict:
    ids = np.asarray(token_adapter)
    ids = ids[ids >= 0]
    out: dict = {}
    for a, n in zip(*np.unique(ids, return_counts=True)):
        r = int(ranks[a])
        out[r] = out.get(r, 0) + int(n)
    return out


def bgmv_bytes(token_adapter, ranks, h_in: int, h_out: int, esize: int) -> int:
    """Minimum HBM bytes of y += s (x A) B with per-token adapters: every
    distinct adapter's pages once, x once, y read and written once."""
    ids = np.asarray(token_adapter)
    T = len(ids)
    used = np.unique(ids[ids >= 0])
    pages = sum(adapter_bytes(int(ranks[a]), h_in, h_out, esize) for a in used)
    return int(pages + T * h_in * esize + 2 * T * h_out * esize)


def shrink_bytes(token_adapter, ranks, h_in: int, esize: int, ld_v: int) -> int:
    """x once, each distinct adapter's A_T once, v written (fp32, rank columns)."""
    ids = np.asarray(token_adapter)
    used = np.unique(ids[ids >= 0])
    a_bytes = sum(int(ranks[a]) * h_in * esize for a in used)
    v_bytes = sum(4 * int(ranks[a]) for a in ids[ids >= 0])
    return int(len(ids) * h_in * esize + a_bytes + v_bytes)


def expand_bytes(token_adapter, ranks, h_out: int, esize: int) -> int:
    """v read, each distinct adapter's B once, y read and written."""
    ids = np.asarray(token_adapter)
    used = np.unique(ids[ids >= 0])
    b_bytes = sum(int(ranks[a]) * h_out * esize for a in used)
    v_bytes = sum(4 * int(ranks[a]) for a in ids[ids >= 0])
    return int(2 * len(ids) * h_out * esize + b_bytes + v_bytes)


def layer_flops(token_adapter, ranks, h_in: int, h_out: int) -> int:
    """Base product plus the adapter term for every adapted token."""
    T = len(token_adapter)
    return base_flops(T, h_in, h_out) + adapter_flops(tokens_per_rank(token_adapter, ranks), h_in, h_out)
