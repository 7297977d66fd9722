"""Helpers for GPU-vs-oracle parity tests.

Tolerances (max |gpu - oracle| / max |oracle| over one output tensor):
  * outputs stored in bf16 (bf16 inputs, fp32 accumulation): 2e-2;
  * outputs stored in fp32 from fp32 inputs: 1e-5;
  * v (fp32) from bf16 inputs: 1e-4 -- exact bf16 products summed in fp32
    over at most a few thousand terms stay orders of magnitude below this.
Integer probes are compared bit for bit.
"""
from __future__ import annotations

import numpy as np

import oracle
from segmented_gathered_rank_gb300 import inputs as I

TOL_Y = {I.BF16: 2e-2, I.F32: 1e-5}
TOL_V = {I.BF16: 1e-4, I.F32: 1e-5}


def rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    diff = np.max(np.abs(got - ref)) if ref.size else 0.0
    return float(diff / scale) if scale > 0 else float(diff)


def token_ids(w: I.Workload) -> np.ndarray:
    """Per-token adapter ids, derived by the oracle from the segment table."""
    st, tok = oracle.token_adapters(w.seg_starts, w.seg_adapter, w.T)
    assert st == 0
    return tok


def oracle_delta(w: I.Workload, m: int, y0, rows=None, W=None, layer: int = 0, ids=None):
    """Oracle y for the listed rows: y0 (+ x.W^T if W) + adapter term."""
    tok = token_ids(w)
    ad = oracle.adapters_for(w, m, ids=ids, layer=layer)
    x = w.x(m, layer)
    rows = np.arange(w.T, dtype=np.int32) if rows is None else np.asarray(rows, np.int32)
    y0r = np.zeros((len(rows), w.matrices[m].h_out)) if y0 is None else np.asarray(y0)[rows]
    y, st = oracle.layer(x, W, tok, ad, w.matrices[m].h_out, y0=y0r, rows=rows)
    return y, st


def oracle_v(w: I.Workload, m: int, ld_v: int, rows=None, layer: int = 0, ids=None):
    tok = token_ids(w)
    ad = oracle.adapters_for(w, m, ids=ids, layer=layer)
    v, st = oracle.shrink(w.x(m, layer), tok, ad, ld_v, rows=rows)
    return v, st


def written_mask(w: I.Workload, ld_v: int, rows=None) -> np.ndarray:
    """Entries of v the shrink defines: j < rank of the token's (valid) adapter."""
    tok = token_ids(w)
    rows = np.arange(w.T) if rows is None else np.asarray(rows)
    mask = np.zeros((len(rows), ld_v), bool)
    for i, t in enumerate(rows):
        a = tok[t]
        if 0 <= a < w.n_adapters:
            mask[i, : int(w.ranks[a])] = True
    return mask


def sample_rows(w: I.Workload, n_random: int, seed: int = 0) -> np.ndarray:
    """Segment first/last tokens plus random tokens, sorted and unique."""
    rng = np.random.default_rng(seed)
    picks = set()
    for s in range(w.S):
        lo, hi = int(w.seg_starts[s]), int(w.seg_starts[s + 1])
        if hi > lo:
            picks.update({lo, hi - 1})
    picks.update(rng.integers(0, w.T, n_random).tolist())
    return np.array(sorted(picks), np.int32)
