"""Seeded synthetic inputs for the multi-LoRA mixed-batch adapter update.

Data only.  This module draws activations, base weights, adapter weights, ranks,
scales, segment tables and adapter ids for the workloads the library is tested
and measured on.  It holds none of the method's arithmetic: no shrink, no
expand, no base product, no mapping of segments onto tokens.  Both sides of a
parity check (the CUDA library and the CPU oracle) read what it returns.

Every tensor is drawn from its own numpy ``default_rng`` stream, keyed by
``[seed, kind, ...]``, so any single tensor (one adapter of one layer, one
layer's activations) can be regenerated on its own.  Normal distributions are
written N(mean, variance), as in the workload descriptions; numpy is given the
standard deviation.  bf16 workloads draw in fp32 and round to bf16 with
round-to-nearest-even; the arrays returned are float32 holding exactly the
bf16 values, so widening them to float64 for the oracle is exact.

Workloads (the adapter update of "Multi-LoRA Serving - S-LoRA/Punica
Batching...", section "The kernel trick: gather, do not merge"):

* ``tiny_sgmv``           4 adapters, rank 8, h 256, fp32, 64 tokens in
                          segments of 16/40/8 with adapters 0/2/3.
* ``decode_bgmv``         256 decode tokens, adapter ids uniform over 32,
                          4096 -> 4096, rank 16, bf16.
* ``prefill_sgmv``        16 segments, Zipf(1.2) lengths capped at 2048 and
                          summing to 8192, 16 distinct adapters of 64,
                          4096 -> 4096 (q, o) and 4096 -> 1024 (k, v), bf16.
* ``encoder_mixed_rank``  1024 adapters x 48 matrices (12 layers x q/k/v/o,
                          768 -> 768), ranks from {8,16,32,64} with
                          probabilities {.4,.3,.2,.1}, 128 sequences x 128
                          tokens with Zipf(1.1) adapter ids, pages of 768.
* ``fused_layer``         4 prefill segments of 1024 tokens + 512 decode
                          tokens, q/k/v/o of a 4096-wide layer, 128 adapters
                          with Zipf(1.0) traffic, rank 16 except adapter 0 at
                          rank 128, base weights N(0, 1/4096).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32 = "f32"
BF16 = "bf16"

# Stream kinds for the per-tensor generators.
_K_IDS, _K_X, _K_Y0, _K_W, _K_ADAPTER, _K_RANKS, _K_XO = range(7)


# ----------------------------------------------------------------------------
# bf16 helpers (storage format only)
# ----------------------------------------------------------------------------
def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (u.astype(np.uint32) << 16).view(np.float32).reshape(a.shape)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """The uint16 bf16 encodings of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("values are not bf16-representable; round them first")
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen uint16 bf16 encodings to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), *[int(k) for k in key]])


def _store(a: np.ndarray, dtype: str) -> np.ndarray:
    a = np.asarray(a, dtype=np.float32)
    return round_to_bf16(a) if dtype == BF16 else np.ascontiguousarray(a)


# ----------------------------------------------------------------------------
# Distributions
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Dist:
    """A value distribution: ``normal`` with ``variance``, or ``uniform`` on [-half, half]."""
    kind: str
    param: float

    def draw(self, rng: np.random.Generator, shape) -> np.ndarray:
        if self.kind == "normal":
            return rng.normal(0.0, np.sqrt(self.param), shape).astype(np.float32)
        if self.kind == "uniform":
            return rng.uniform(-self.param, self.param, shape).astype(np.float32)
        if self.kind == "zero":
            return np.zeros(shape, np.float32)
        raise ValueError(self.kind)


def normal(variance: float) -> Dist:
    return Dist("normal", float(variance))


def uniform(half_width: float) -> Dist:
    return Dist("uniform", float(half_width))


ZERO = Dist("zero", 0.0)


@dataclass(frozen=True)
class Matrix:
    """One adapted projection: name and its input/output widths."""
    name: str
    h_in: int
    h_out: int


@dataclass
class Workload:
    """A synthetic mixed batch and the adapter population it draws on.

    ``seg_starts`` (S+1) and ``seg_adapter`` (S) describe the batch as runs of
    tokens sharing an adapter.  For decode batches, ``token_adapter`` holds
    the drawn per-token ids and each token is a segment of length one.
    Adapter ids ``0..n_adapters-1`` exist for every matrix, with rank
    ``ranks[a]`` and scale ``scales[a]`` (the same for every matrix).
    """
    name: str
    dtype: str
    T: int
    matrices: list
    n_adapters: int
    ranks: np.ndarray
    scales: np.ndarray
    seg_starts: np.ndarray
    seg_adapter: np.ndarray
    page_elems: int
    max_rank: int
    seed: int
    x_dist: Dist
    a_dist: Dist
    b_dist: Dist
    w_dist: Dist
    y0_dist: Dist = field(default_factory=lambda: normal(1.0))
    token_adapter: np.ndarray | None = None
    shared_x: dict = field(default_factory=dict)   # matrix index -> activation stream id
    layers: int = 1                                  # distinct copies (bench rotation)
    probe: bool = False                              # small-integer values (see integer_probe)
    zero_b: tuple = ()                               # adapters whose B is all zeros (A_T drawn as usual)

    # -- tensors ----------------------------------------------------------
    def x(self, m: int = 0, layer: int = 0) -> np.ndarray:
        """Activations [T x h_in] feeding matrix ``m`` of copy ``layer``."""
        mat = self.matrices[m]
        stream = self.shared_x.get(m, m)
        if self.probe:
            return probe_x(self.seed + 1000 * layer + stream, self.T, mat.h_in)
        return _store(self.x_dist.draw(_rng(self.seed, _K_X, layer, stream), (self.T, mat.h_in)), self.dtype)

    def y0(self, m: int = 0, layer: int = 0) -> np.ndarray:
        """Initial output [T x h_out] that the adapter update adds to."""
        mat = self.matrices[m]
        if self.probe:
            return probe_y0(self.seed + 1000 * layer + m, self.T, mat.h_out)
        return _store(self.y0_dist.draw(_rng(self.seed, _K_Y0, layer, m), (self.T, mat.h_out)), self.dtype)

    def W(self, m: int = 0, layer: int = 0) -> np.ndarray:
        """Base weight [h_out x h_in] (row n holds output feature n)."""
        mat = self.matrices[m]
        if self.probe:
            return probe_w(self.seed + 1000 * layer + m, mat.h_out, mat.h_in)
        return _store(self.w_dist.draw(_rng(self.seed, _K_W, layer, m), (mat.h_out, mat.h_in)), self.dtype)

    def W_e4m3(self, m: int = 0, layer: int = 0):
        """The base weight of matrix m as an FP8 base would hold it: e4m3 codes
        [h_out x h_in] (uint8) of W / s_w and the per-tensor scale s_w =
        max|W| / 448 (float32).  Input preparation of the caller's side; the
        codes come from torch's float8_e4m3fn conversion (every value is within
        +-448 by the choice of s_w)."""
        import torch
        w = np.asarray(self.W(m, layer), np.float32)
        amax = np.float32(np.max(np.abs(w)))
        s_w = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
        codes = torch.from_numpy(np.ascontiguousarray(w / s_w, np.float32)).to(torch.float8_e4m3fn)
        return codes.view(torch.uint8).numpy().copy(), float(s_w)

    def adapter(self, a: int, m: int = 0, layer: int = 0):
        """(A_T [r x h_in], B [r x h_out]) of adapter ``a`` on matrix ``m``.

        Row j of A_T is column j of A_a (so x.A_a is x against each row of
        A_T); row j of B is row j of B_a.
        """
        mat = self.matrices[m]
        r = int(self.ranks[a])
        if self.probe:
            at, b = probe_adapter(self.seed + 1000 * layer + m, a, r, mat.h_in, mat.h_out)
        else:
            rng = _rng(self.seed, _K_ADAPTER, layer, m, a)
            at = _store(self.a_dist.draw(rng, (r, mat.h_in)), self.dtype)
            b = _store(self.b_dist.draw(rng, (r, mat.h_out)), self.dtype)
        if a in self.zero_b:
            b = np.zeros_like(b)
        return at, b

    @property
    def S(self) -> int:
        return len(self.seg_adapter)

    def used_adapters(self) -> np.ndarray:
        ids = self.seg_adapter if self.token_adapter is None else self.token_adapter
        ids = np.asarray(ids)
        return np.unique(ids[ids >= 0])


# ----------------------------------------------------------------------------
# Samplers used by the workload recipes
# ----------------------------------------------------------------------------
def bounded_zipf(rng: np.random.Generator, n: int, s: float, size: int) -> np.ndarray:
    """Ids 0..n-1 with P(id = k-1) proportional to k^-s, by inverse CDF.

    Same sampler as the adapter-cache simulation on "Multi-LoRA Serving"
    (section "Memory: slots, tiers and paging"): cumulative normalised
    weights, then the first index whose CDF reaches the uniform draw.
    """
    w = 1.0 / np.power(np.arange(1, n + 1, dtype=np.float64), s)
    cdf = np.cumsum(w / w.sum())
    u = rng.random(size)
    return np.minimum(np.searchsorted(cdf, u, side="left"), n - 1).astype(np.int32)


def lcg_uniforms(seed: int, n: int) -> np.ndarray:
    """The linear congruential generator of the adapter-cache simulation on
    "Multi-LoRA Serving" (section "Memory: slots, tiers and paging"): state
    s <- (1664525 s + 1013904223) mod 2^32 starting from ``seed``, each step
    yielding s / 2^32 in [0, 1).  Exact integer arithmetic."""
    out = np.empty(n, np.float64)
    s = seed & 0xFFFFFFFF
    for i in range(n):
        s = (s * 1664525 + 1013904223) & 0xFFFFFFFF
        out[i] = s / 4294967296.0
    return out


def adapter_request_trace(n_adapters: int = 500, requests: int = 50_000, s: float = 1.1,
                          seed: int = 11) -> np.ndarray:
    """Adapter ids of a request stream with Zipf(s) popularity, drawn as the
    page's adapter-cache simulation draws them: weights 1 / (i+1)^s for ids
    i = 0..n-1, a cumulative distribution built by adding the normalised
    weights left to right (the total itself summed left to right), and for
    each LCG uniform u the first id whose cumulative value is >= u.  The
    defaults are that simulation's workload (500 adapters, 50,000 requests,
    s = 1.1, LCG seed 11)."""
    w = [1.0 / float(i + 1) ** s for i in range(n_adapters)]
    total = 0.0
    for v in w:
        total += v
    cdf = np.empty(n_adapters, np.float64)
    acc = 0.0
    for i, v in enumerate(w):
        acc = acc + v / total
        cdf[i] = acc
    u = lcg_uniforms(seed, requests)
    ids = np.searchsorted(cdf, u, side="left")
    return np.minimum(ids, n_adapters - 1).astype(np.int32)


def zipf_lengths(n: int, s: float, total: int, cap: int) -> np.ndarray:
    """Deterministic segment lengths L_k ~ k^-s (k=1..n), capped, summing to ``total``.

    Lengths above ``cap`` are pinned at ``cap`` and the remainder is shared
    again in proportion (water-filling); fractional parts are resolved by
    largest remainder.
    """
    w = np.arange(1, n + 1, dtype=np.float64) ** (-s)
    fixed = np.zeros(n, bool)
    L = np.zeros(n)
    while True:
        free = ~fixed
        rem = total - cap * fixed.sum()
        L[free] = rem * w[free] / w[free].sum()
        L[fixed] = cap
        over = free & (L > cap)
        if not over.any():
            break
        fixed |= over
    out = np.floor(L).astype(np.int64)
    short = int(total - out.sum())
    order = np.argsort(-(L - out), kind="stable")
    out[order[:short]] += 1
    return out.astype(np.int32)


def _segments_from_lengths(lengths) -> np.ndarray:
    starts = np.zeros(len(lengths) + 1, np.int32)
    starts[1:] = np.cumsum(np.asarray(lengths, np.int64))
    return starts


def _unit_segments(T: int) -> np.ndarray:
    return np.arange(T + 1, dtype=np.int32)


# ----------------------------------------------------------------------------
# The five workloads
# ----------------------------------------------------------------------------
def tiny_sgmv(seed: int = 0) -> Workload:
    lengths, ids = [16, 40, 8], [0, 2, 3]
    return Workload(
        name="tiny_sgmv", dtype=F32, T=64, matrices=[Matrix("proj", 256, 256)],
        n_adapters=4, ranks=np.full(4, 8, np.int32), scales=np.full(4, 2.0, np.float32),
        seg_starts=_segments_from_lengths(lengths), seg_adapter=np.array(ids, np.int32),
        page_elems=256, max_rank=8, seed=seed,
        x_dist=normal(1.0), a_dist=normal(1 / 256), b_dist=normal(0.02), w_dist=normal(1 / 256))


def decode_bgmv(seed: int = 0, layers: int = 1) -> Workload:
    T, n = 256, 32
    ids = _rng(seed, _K_IDS).integers(0, n, T).astype(np.int32)
    return Workload(
        name="decode_bgmv", dtype=BF16, T=T, matrices=[Matrix("q_proj", 4096, 4096)],
        n_adapters=n, ranks=np.full(n, 16, np.int32), scales=np.full(n, 2.0, np.float32),
        seg_starts=_unit_segments(T), seg_adapter=ids.copy(), token_adapter=ids,
        page_elems=4096, max_rank=16, seed=seed,
        x_dist=normal(1.0), a_dist=uniform(1 / 64), b_dist=normal(0.01), w_dist=normal(1 / 4096),
        layers=layers)


def prefill_sgmv(seed: int = 0, layers: int = 1) -> Workload:
    lengths = zipf_lengths(16, 1.2, 8192, 2048)
    ids = _rng(seed, _K_IDS).choice(64, 16, replace=False).astype(np.int32)
    mats = [Matrix("q_proj", 4096, 4096), Matrix("k_proj", 4096, 1024),
            Matrix("v_proj", 4096, 1024), Matrix("o_proj", 4096, 4096)]
    return Workload(
        name="prefill_sgmv", dtype=BF16, T=8192, matrices=mats,
        n_adapters=64, ranks=np.full(64, 16, np.int32), scales=np.full(64, 2.0, np.float32),
        seg_starts=_segments_from_lengths(lengths), seg_adapter=ids,
        page_elems=4096, max_rank=16, seed=seed,
        x_dist=normal(1.0), a_dist=uniform(1 / 64), b_dist=normal(0.01), w_dist=normal(1 / 4096),
        shared_x={0: 0, 1: 0, 2: 0, 3: 3}, layers=layers)


def encoder_mixed_rank(seed: int = 0) -> Workload:
    n, n_layers, seqs, seq_len = 1024, 12, 128, 128
    ranks = _rng(seed, _K_RANKS).choice(np.array([8, 16, 32, 64]), n, p=[0.4, 0.3, 0.2, 0.1]).astype(np.int32)
    ids = bounded_zipf(_rng(seed, _K_IDS), n, 1.1, seqs)
    mats = [Matrix(f"layer{l}.{p}", 768, 768) for l in range(n_layers) for p in ("q", "k", "v", "o")]
    return Workload(
        name="encoder_mixed_rank", dtype=BF16, T=seqs * seq_len, matrices=mats,
        n_adapters=n, ranks=ranks, scales=np.full(n, 2.0, np.float32),
        seg_starts=_segments_from_lengths([seq_len] * seqs), seg_adapter=ids,
        page_elems=768, max_rank=64, seed=seed,
        x_dist=normal(1.0), a_dist=uniform(1 / 64), b_dist=normal(0.01), w_dist=normal(1 / 768))


def fused_layer(seed: int = 0, layers: int = 1) -> Workload:
    n = 128
    ranks = np.full(n, 16, np.int32)
    ranks[0] = 128
    draws = bounded_zipf(_rng(seed, _K_IDS), n, 1.0, 4 + 512)
    lengths = [1024] * 4 + [1] * 512
    mats = [Matrix("q_proj", 4096, 4096), Matrix("k_proj", 4096, 1024),
            Matrix("v_proj", 4096, 1024), Matrix("o_proj", 4096, 4096)]
    return Workload(
        name="fused_layer", dtype=BF16, T=4608, matrices=mats,
        n_adapters=n, ranks=ranks, scales=np.full(n, 2.0, np.float32),
        seg_starts=_segments_from_lengths(lengths), seg_adapter=draws,
        page_elems=4096, max_rank=128, seed=seed,
        x_dist=normal(1.0), a_dist=uniform(1 / 64), b_dist=normal(0.01), w_dist=normal(1 / 4096),
        shared_x={0: 0, 1: 0, 2: 0, 3: 3}, layers=layers)


WORKLOADS = {
    "tiny_sgmv": tiny_sgmv,
    "decode_bgmv": decode_bgmv,
    "prefill_sgmv": prefill_sgmv,
    "encoder_mixed_rank": encoder_mixed_rank,
    "fused_layer": fused_layer,
}


# ----------------------------------------------------------------------------
# Small randomized cases for parity tests
# ----------------------------------------------------------------------------
def random_case(seed: int, T: int, lengths=None, h_in: int = 256, h_out: int = 256,
                n_adapters: int = 6, ranks=None, dtype: str = BF16, page_elems: int | None = None,
                none_fraction: float = 0.0, decode: bool = False,
                x_dist: Dist = normal(1.0), a_dist: Dist = uniform(1 / 16),
                b_dist: Dist = normal(0.01), w_dist: Dist | None = None) -> Workload:
    """A small mixed batch with ragged segments, ragged ranks and optional
    tokens without an adapter (id -1).

    ``lengths`` may contain zeros (empty segments).  With ``decode`` every
    token is its own segment and ``token_adapter`` is filled.
    """
    rng = _rng(seed, _K_IDS)
    if ranks is None:
        ranks = rng.choice(np.array([8, 16, 32]), n_adapters)
    ranks = np.asarray(ranks, np.int32)
    n_adapters = len(ranks)
    if decode:
        lengths = [1] * T
    elif lengths is None:
        cuts = np.sort(rng.integers(0, T + 1, max(1, T // 37)))
        lengths = np.diff(np.concatenate([[0], cuts, [T]])).tolist()
    lengths = np.asarray(lengths, np.int64)
    assert lengths.sum() == T
    ids = rng.integers(0, n_adapters, len(lengths)).astype(np.int32)
    if none_fraction > 0:
        ids[rng.random(len(ids)) < none_fraction] = -1
    max_rank = int(ranks.max()) if len(ranks) else 0
    w = Workload(
        name=f"random{seed}", dtype=dtype, T=T, matrices=[Matrix("proj", h_in, h_out)],
        n_adapters=n_adapters, ranks=ranks, scales=rng.choice(np.array([0.5, 1.0, 2.0], np.float32), n_adapters),
        seg_starts=_segments_from_lengths(lengths), seg_adapter=ids,
        page_elems=page_elems or max(h_in, h_out), max_rank=max(max_rank, 1), seed=seed,
        x_dist=x_dist, a_dist=a_dist, b_dist=b_dist, w_dist=w_dist or normal(1.0 / h_in))
    if decode:
        w.token_adapter = ids.copy()
    return w


def integer_probe(seed: int, T: int, lengths, h_in: int, h_out: int, ranks, dtype: str = BF16,
                  none_fraction: float = 0.0) -> Workload:
    """Small-integer activations and adapters whose every partial sum is exact.

    x has three entries in {-1, 1} per row and zeros elsewhere; A_T, B and W
    hold integers in {-2..2} with most entries zero.  With |x.A| and the
    outputs bounded well inside bf16's exact integers, every summation order
    gives the same result, so a correct kernel matches the oracle bit for bit.
    """
    rng = _rng(seed, _K_IDS)
    ranks = np.asarray(ranks, np.int32)
    lengths = np.asarray(lengths, np.int64)
    ids = rng.integers(0, len(ranks), len(lengths)).astype(np.int32)
    if none_fraction > 0:
        ids[rng.random(len(ids)) < none_fraction] = -1
    w = Workload(
        name=f"intprobe{seed}", dtype=dtype, T=T, matrices=[Matrix("proj", h_in, h_out)],
        n_adapters=len(ranks), ranks=ranks, scales=rng.choice(np.array([1.0, 2.0], np.float32), len(ranks)),
        seg_starts=_segments_from_lengths(lengths), seg_adapter=ids,
        page_elems=max(h_in, h_out), max_rank=int(ranks.max()), seed=seed,
        x_dist=ZERO, a_dist=ZERO, b_dist=ZERO, w_dist=ZERO, y0_dist=ZERO, probe=True)
    return w


def probe_x(seed: int, T: int, h_in: int, nnz: int = 3) -> np.ndarray:
    rng = _rng(seed, _K_X)
    x = np.zeros((T, h_in), np.float32)
    for t in range(T):
        cols = rng.choice(h_in, nnz, replace=False)
        x[t, cols] = rng.choice(np.array([-1.0, 1.0], np.float32), nnz)
    return x


def probe_adapter(seed: int, a: int, r: int, h_in: int, h_out: int, density: float = 0.05):
    rng = _rng(seed, _K_ADAPTER, a)
    at = rng.integers(-2, 3, (r, h_in)).astype(np.float32) * (rng.random((r, h_in)) < density)
    b = rng.integers(-2, 3, (r, h_out)).astype(np.float32) * (rng.random((r, h_out)) < density)
    return np.ascontiguousarray(at), np.ascontiguousarray(b)


def probe_y0(seed: int, T: int, h_out: int) -> np.ndarray:
    rng = _rng(seed, _K_Y0)
    return rng.integers(-4, 5, (T, h_out)).astype(np.float32)


def probe_w(seed: int, h_out: int, h_in: int, density: float = 0.02) -> np.ndarray:
    rng = _rng(seed, _K_W)
    w = rng.integers(-2, 3, (h_out, h_in)).astype(np.float32) * (rng.random((h_out, h_in)) < density)
    return np.ascontiguousarray(w)


# ----------------------------------------------------------------------------
# The worked example printed on "Multi-LoRA Serving" (numpy listing)
# ----------------------------------------------------------------------------
def page_example():
    """Inputs of the page's numpy example, drawn in the page's order.

    d=2048, r=16, 50 adapters, batch 64, scale 2, generator seed 0: W, then
    the stacked A (r x d each), the stacked B (d x r each), X, then one
    adapter id per request.  The page prints that this batch touches 34
    distinct adapters; reproducing that count needs the same draw order.
    Returned in this library's convention: A_T[a] = A[a] (r x d) and
    B[a] = the page's B[a] transposed (r x d).
    """
    rng = np.random.default_rng(0)
    d, r, n, batch, scale = 2048, 16, 50, 64, 2.0
    W = rng.normal(0, 0.02, (d, d)).astype(np.float32)
    A = rng.normal(0, 0.02, (n, r, d)).astype(np.float32)
    Bp = rng.normal(0, 0.02, (n, d, r)).astype(np.float32)
    X = rng.normal(0, 1, (batch, d)).astype(np.float32)
    ids = rng.integers(0, n, batch)
    return dict(d=d, r=r, n=n, batch=batch, scale=scale, W=W, A_T=A,
                B=np.ascontiguousarray(np.transpose(Bp, (0, 2, 1))), X=X, ids=ids.astype(np.int32))
