"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each ``check_*`` takes a loaded oracle library and raises AssertionError when
the oracle disagrees with the pin.  ``tests/test_oracle.py`` runs them on the
real oracle; ``tests/test_oracle_mutants.py`` runs them on copies of the
oracle with a planted mistake (in a subprocess, through ``main`` below) and
expects at least one to fail.

None of these re-types the oracle's loops.  The pins are:
  * the worked example on "Multi-LoRA Serving" (numpy listing and its printed
    output): with the page's inputs, merged-per-adapter weights and the
    gathered low-rank form agree (allclose, atol 1e-3) and the batch holds 34
    distinct adapters;
  * the merge identity W' = W + A B (S-LoRA slide 5, and the page's
    "merge-per-adapter" option), evaluated as a merged-weight product;
  * rank 0 and zero B leave the base output unchanged, exactly;
  * permuting segments permutes output rows, exactly;
  * brute force on tiny inputs, by pure-Python loops over an explicit merged
    weight per token;
  * integer one-hot probes whose outputs are known in closed form;
  * shrink and expand against numpy's matrix product on small data;
  * the segment table semantics, by brute force over token indices.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import oracle  # noqa: E402
from segmented_gathered_rank_gb300 import inputs  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_example.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _merged_rows(x_rows, W, at, b, s):
    """x . (W + s * A B)^T with the merged weight formed first (fp64)."""
    Wm = W.astype(np.float64) + s * (b.astype(np.float64).T @ at.astype(np.float64))
    return x_rows.astype(np.float64) @ Wm.T


# ----------------------------------------------------------------------------
def check_page_example(lib):
    g = _golden()
    ex = inputs.page_example()
    ids = ex["ids"]
    assert len(np.unique(ids)) == g["distinct_adapters"], "distinct adapter count differs from the page"
    n = ex["n"]
    ad = oracle.Adapters(n, {a: (ex["r"], ex["scale"], ex["A_T"][a], ex["B"][a]) for a in range(n)})
    y, st = oracle.layer(ex["X"], ex["W"], ids, ad, ex["d"], lib=lib)
    assert st == 0
    # The page's merge-per-adapter option: group rows by adapter, merge, multiply.
    y1 = np.empty_like(y)
    for a in np.unique(ids):
        rows = ids == a
        y1[rows] = _merged_rows(ex["X"][rows], ex["W"], ex["A_T"][a], ex["B"][a], ex["scale"])
    assert np.allclose(y1, y, atol=g["atol"]) == g["same_outputs"]
    # In double precision the two forms agree to rounding.
    assert np.max(np.abs(y1 - y)) <= 1e-9 * max(1.0, np.max(np.abs(y1)))


def check_merged_invariant(lib):
    for seed in range(3):
        w = inputs.random_case(seed, T=45, h_in=40, h_out=24, n_adapters=5, ranks=[1, 3, 7, 2, 5],
                               dtype=inputs.F32, lengths=[7, 0, 20, 1, 17], w_dist=inputs.normal(0.1),
                               b_dist=inputs.normal(0.5), a_dist=inputs.normal(0.5))
        x, W = w.x(), w.W()
        ad = oracle.adapters_for(w, ids=range(w.n_adapters))
        st, tok = oracle.token_adapters(w.seg_starts, w.seg_adapter, w.T, lib=lib)
        assert st == 0
        y, st = oracle.layer(x, W, tok, ad, 24, lib=lib)
        assert st == 0
        for s in range(w.S):
            lo, hi = w.seg_starts[s], w.seg_starts[s + 1]
            a = int(w.seg_adapter[s])
            at, b = w.adapter(a)
            ref = _merged_rows(x[lo:hi], W, at, b, float(w.scales[a]))
            assert np.allclose(y[lo:hi], ref, rtol=1e-12, atol=1e-12), f"segment {s}"


def check_rank0_and_zero_b(lib):
    rng = np.random.default_rng(5)
    T, h_in, h_out = 12, 16, 10
    x = rng.normal(size=(T, h_in))
    W = rng.normal(size=(h_out, h_in))
    y0 = rng.normal(size=(T, h_out))
    tok = np.array([0, 1, 1, 0, 2, 2, 2, 0, 1, 2, 0, 1], np.int32)
    ad = oracle.Adapters(3, {0: (0, 2.0, np.zeros((0, h_in)), np.zeros((0, h_out))),
                             1: (4, 2.0, rng.normal(size=(4, h_in)), np.zeros((4, h_out))),
                             2: (3, 0.5, rng.normal(size=(3, h_in)), np.zeros((3, h_out)))})
    none = np.full(T, -1, np.int32)
    y_base, st0 = oracle.layer(x, W, none, ad, h_out, y0=y0, lib=lib)
    y_adapt, st1 = oracle.layer(x, W, tok, ad, h_out, y0=y0, lib=lib)
    assert st0 == 0 and st1 == 0
    assert np.array_equal(y_base, y_adapt)
    # Without a base: the update leaves y0 exactly as it was.
    y_d, st = oracle.layer(x, None, tok, ad, h_out, y0=y0, lib=lib)
    assert st == 0 and np.array_equal(y_d, y0)
    v, st = oracle.shrink(x, tok, ad, 4, lib=lib)
    y_e, st2 = oracle.expand(np.nan_to_num(v), tok, ad, y0, lib=lib)
    assert st == 0 and st2 == 0 and np.array_equal(y_e, y0)


def check_permutation(lib):
    w = inputs.random_case(11, T=60, h_in=32, h_out=24, n_adapters=4, ranks=[2, 5, 3, 4],
                           dtype=inputs.F32, lengths=[9, 14, 0, 21, 16])
    x, W = w.x(), w.W()
    ad = oracle.adapters_for(w, ids=range(w.n_adapters))
    _, tok = oracle.token_adapters(w.seg_starts, w.seg_adapter, w.T, lib=lib)
    y, _ = oracle.layer(x, W, tok, ad, 24, lib=lib)
    perm = np.array([3, 0, 4, 2, 1])
    lens = np.diff(w.seg_starts)[perm]
    starts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rows = np.concatenate([np.arange(w.seg_starts[s], w.seg_starts[s + 1]) for s in perm]).astype(np.int64)
    _, tok2 = oracle.token_adapters(starts, w.seg_adapter[perm], w.T, lib=lib)
    y2, _ = oracle.layer(x[rows], W, tok2, ad, 24, lib=lib)
    assert np.array_equal(y2, y[rows])


def check_brute_force_tiny(lib):
    rng = np.random.default_rng(7)
    for trial in range(4):
        T, h_in, h_out = 6, 5 + trial, 4 + trial
        n = 3
        ranks = [1 + (trial + a) % 4 for a in range(n)]
        scales = [0.5, 2.0, -1.5]
        ats = [rng.normal(size=(r, h_in)) for r in ranks]
        bs = [rng.normal(size=(r, h_out)) for r in ranks]
        x = rng.normal(size=(T, h_in)).tolist()
        W = rng.normal(size=(h_out, h_in)).tolist()
        tok = [int(v) for v in rng.integers(-1, n, T)]
        y_bf = []
        for t in range(T):
            # merged weight for this token, written element by element
            Wt = [[W[o][k] for k in range(h_in)] for o in range(h_out)]
            a = tok[t]
            if a >= 0:
                for o in range(h_out):
                    for k in range(h_in):
                        Wt[o][k] += scales[a] * sum(bs[a][j][o] * ats[a][j][k] for j in range(ranks[a]))
            y_bf.append([sum(Wt[o][k] * x[t][k] for k in range(h_in)) for o in range(h_out)])
        ad = oracle.Adapters(n, {a: (ranks[a], scales[a], ats[a], bs[a]) for a in range(n)})
        y, st = oracle.layer(np.array(x), np.array(W), np.array(tok, np.int32), ad, h_out, lib=lib)
        assert st == 0
        assert np.allclose(y, np.array(y_bf), rtol=1e-12, atol=1e-12)


def check_integer_onehot(lib):
    # x[t] = c_t * e_{k_t}; A_T_a[j][k] = (j+1) * (k+1) (mod 5) - 2; B_a[j][n] = (a+1) at n == a + j
    # Then v[t][j] = c_t * A_T_a[j][k_t] and y[t][n] = s_a * v[t][n-a] * (a+1) for a <= n < a + r.
    T, h_in, h_out, n = 20, 9, 16, 4
    ranks = [3, 2, 4, 1]
    scales = [1.0, 2.0, 3.0, 0.5]
    rng = np.random.default_rng(3)
    k_t = rng.integers(0, h_in, T)
    c_t = rng.integers(1, 4, T)
    tok = rng.integers(0, n, T).astype(np.int32)
    x = np.zeros((T, h_in))
    x[np.arange(T), k_t] = c_t
    ents = {}
    for a in range(n):
        r = ranks[a]
        at = np.array([[((j + 1) * (k + 1)) % 5 - 2 for k in range(h_in)] for j in range(r)], float)
        b = np.zeros((r, h_out))
        for j in range(r):
            b[j, a + j] = a + 1
        ents[a] = (r, scales[a], at, b)
    ad = oracle.Adapters(n, ents)
    y, st = oracle.layer(x, None, tok, ad, h_out, lib=lib)
    assert st == 0
    for t in range(T):
        a = int(tok[t])
        expect = np.zeros(h_out)
        for j in range(ranks[a]):
            expect[a + j] = scales[a] * c_t[t] * ((((j + 1) * (k_t[t] + 1)) % 5) - 2) * (a + 1)
        assert np.array_equal(y[t], expect), t
    v, st = oracle.shrink(x, tok, ad, 4, lib=lib)
    assert st == 0
    for t in range(T):
        a = int(tok[t])
        for j in range(ranks[a]):
            assert v[t, j] == c_t[t] * ((((j + 1) * (k_t[t] + 1)) % 5) - 2)


def check_shrink_expand_numpy(lib):
    w = inputs.random_case(21, T=33, h_in=48, h_out=40, n_adapters=3, ranks=[4, 8, 2],
                           dtype=inputs.F32, lengths=[10, 3, 20], none_fraction=0.0)
    x = w.x().astype(np.float64)
    y0 = w.y0().astype(np.float64)
    ad = oracle.adapters_for(w, ids=range(w.n_adapters))
    _, tok = oracle.token_adapters(w.seg_starts, w.seg_adapter, w.T, lib=lib)
    v, st = oracle.shrink(x, tok, ad, 8, lib=lib)
    assert st == 0
    y, st = oracle.expand(np.nan_to_num(v), tok, ad, y0, lib=lib)
    assert st == 0
    for a in range(w.n_adapters):
        rows = tok == a
        at, b = w.adapter(a)
        r = int(w.ranks[a])
        vref = np.matmul(x[rows], at.astype(np.float64).T)
        assert np.allclose(v[rows, :r], vref, rtol=1e-12, atol=1e-12)
        assert np.all(np.isnan(v[rows, r:]))
        yref = y0[rows] + float(w.scales[a]) * np.matmul(vref, b.astype(np.float64))
        assert np.allclose(y[rows], yref, rtol=1e-12, atol=1e-12)
    # The two halves compose to the whole layer without a base.
    yl, st = oracle.layer(x, None, tok, ad, w.matrices[0].h_out, y0=y0, lib=lib)
    assert st == 0 and np.allclose(yl, y, rtol=1e-12, atol=1e-12)


def check_segments(lib):
    rng = np.random.default_rng(9)
    for _ in range(20):
        S = int(rng.integers(0, 8))
        lens = rng.integers(0, 6, S)
        T = int(lens.sum())
        starts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        ids = rng.integers(-1, 5, S).astype(np.int32)
        st, tok = oracle.token_adapters(starts, ids, T, lib=lib)
        assert st == 0
        expect = []
        for s in range(S):
            expect += [int(ids[s])] * int(lens[s])
        assert tok.tolist() == expect
    bad = [
        (np.array([1, 3], np.int32), np.array([0], np.int32), 3),        # does not start at 0
        (np.array([0, 3, 2, 5], np.int32), np.array([0, 1, 2], np.int32), 5),  # decreasing
        (np.array([0, 2, 4], np.int32), np.array([0, 1], np.int32), 5),  # does not end at T
    ]
    for starts, ids, T in bad:
        st, _ = oracle.token_adapters(starts, ids, T, lib=lib)
        assert st == oracle.ERR_SEGMENTS


def check_invalid_ids(lib):
    rng = np.random.default_rng(2)
    T, h_in, h_out = 6, 8, 5
    x = rng.normal(size=(T, h_in))
    W = rng.normal(size=(h_out, h_in))
    ad = oracle.Adapters(3, {0: (2, 1.0, rng.normal(size=(2, h_in)), rng.normal(size=(2, h_out)))})
    tok = np.array([0, -1, 1, 7, 0, -3], np.int32)       # 1: not loaded, 7: out of range
    y, st = oracle.layer(x, W, tok, ad, h_out, lib=lib)
    assert st == oracle.ERR_ADAPTER
    base = x @ W.T
    for t in (1, 2, 3, 5):
        assert np.allclose(y[t], base[t], rtol=1e-12, atol=1e-12)
    assert not np.allclose(y[0], base[0])
    # a rank above ld_v is refused by shrink and expand
    v, st = oracle.shrink(x, np.zeros(T, np.int32), ad, 1, lib=lib)
    assert st == oracle.ERR_RANK


CHECKS = [check_page_example, check_merged_invariant, check_rank0_and_zero_b, check_permutation,
          check_brute_force_tiny, check_integer_onehot, check_shrink_expand_numpy, check_segments,
          check_invalid_ids]


def main(argv):
    """Run every check against the oracle library at argv[1]; print a JSON verdict."""
    lib = oracle.load(argv[1])
    out = {}
    for c in CHECKS:
        try:
            c(lib)
            out[c.__name__] = "ok"
        except Exception as e:  # noqa: BLE001 - any failure is a caught mutant
            out[c.__name__] = f"fail: {type(e).__name__}: {e}"[:200]
    print(json.dumps(out))


if __name__ == "__main__":
    main(sys.argv)
