"""The seeded input generators (no GPU): each workload has the shapes, ranks,
segment structure and value distributions its recipe states, the samplers
do what their names say, draws are reproducible per seed, and the bf16
storage helpers round to nearest even."""
import numpy as np
import pytest

from segmented_gathered_rank_gb300 import inputs as I


def _lengths(w):
    return np.diff(np.asarray(w.seg_starts))


def test_tiny_sgmv_recipe():
    w = I.tiny_sgmv()
    assert w.dtype == I.F32 and w.T == 64 and w.n_adapters == 4
    assert list(_lengths(w)) == [16, 40, 8] and list(w.seg_adapter) == [0, 2, 3]
    assert set(w.ranks.tolist()) == {8} and set(w.scales.tolist()) == {2.0}
    assert (w.matrices[0].h_in, w.matrices[0].h_out) == (256, 256)


def test_decode_bgmv_recipe():
    w = I.decode_bgmv()
    assert w.T == 256 and w.n_adapters == 32 and set(w.ranks.tolist()) == {16}
    assert list(_lengths(w)) == [1] * 256                      # one token per segment
    ids = np.asarray(w.token_adapter)
    assert ids.min() >= 0 and ids.max() < 32 and len(np.unique(ids)) > 24
    assert (w.matrices[0].h_in, w.matrices[0].h_out) == (4096, 4096)


def test_prefill_sgmv_recipe():
    w = I.prefill_sgmv()
    L = _lengths(w)
    assert len(L) == 16 and L.sum() == 8192 and L.max() <= 2048
    assert np.all(np.diff(L) <= 0)                             # Zipf: longest first
    assert len(np.unique(w.seg_adapter)) == 16 and w.seg_adapter.max() < 64
    assert [(m.h_in, m.h_out) for m in w.matrices] == [(4096, 4096), (4096, 1024), (4096, 1024), (4096, 4096)]


def test_encoder_recipe():
    w = I.encoder_mixed_rank()
    assert w.T == 128 * 128 and list(_lengths(w)) == [128] * 128
    assert len(w.matrices) == 48 and all((m.h_in, m.h_out) == (768, 768) for m in w.matrices)
    assert w.n_adapters == 1024 and set(np.unique(w.ranks).tolist()) <= {8, 16, 32, 64}
    freq = np.array([(w.ranks == r).mean() for r in (8, 16, 32, 64)])
    assert np.all(np.abs(freq - [0.4, 0.3, 0.2, 0.1]) < 0.05)
    ids = np.asarray(w.seg_adapter)
    assert ids.min() >= 0 and ids.max() < 1024
    assert np.mean(ids < 10) > 0.2                             # Zipf(1.1): the first ids dominate


def test_fused_layer_recipe():
    w = I.fused_layer()
    L = _lengths(w)
    assert w.T == 4608 and list(L[:4]) == [1024] * 4 and list(L[4:]) == [1] * 512
    assert w.n_adapters == 128 and w.ranks[0] == 128 and set(w.ranks[1:].tolist()) == {16}
    assert [(m.h_in, m.h_out) for m in w.matrices] == [(4096, 4096), (4096, 1024), (4096, 1024), (4096, 4096)]


def test_zipf_lengths_sum_cap_and_order():
    for n, s, total, cap in [(16, 1.2, 8192, 2048), (5, 2.0, 100, 60), (7, 0.5, 1000, 1000)]:
        L = I.zipf_lengths(n, s, total, cap)
        assert len(L) == n and L.sum() == total and L.max() <= cap and np.all(np.diff(L) <= 0)


def test_bounded_zipf_range_and_skew():
    ids = I.bounded_zipf(np.random.default_rng(0), 50, 1.0, 200000)
    assert ids.min() >= 0 and ids.max() <= 49
    counts = np.bincount(ids, minlength=50)
    # P(k) ~ 1/k: the first id about twice as frequent as the second, ten times the tenth
    assert 1.8 < counts[0] / counts[1] < 2.2 and 8 < counts[0] / counts[9] < 12


def test_draws_are_reproducible_per_seed():
    a, b, c = I.random_case(7, T=90), I.random_case(7, T=90), I.random_case(8, T=90)
    assert np.array_equal(a.x(), b.x()) and np.array_equal(a.seg_starts, b.seg_starts)
    assert np.array_equal(a.adapter(0)[0], b.adapter(0)[0])
    assert not np.array_equal(a.x(), c.x())


def test_value_distributions():
    w = I.decode_bgmv()
    x = w.x()
    assert abs(float(x.mean())) < 0.01 and abs(float(x.var()) - 1.0) < 0.02    # N(0, 1)
    at, bm = w.adapter(int(w.used_adapters()[0]))
    assert np.abs(at).max() <= 1 / 64 and np.abs(at).max() > 0.9 / 64            # U(-1/64, 1/64)
    assert abs(float(bm.std()) - 0.1) < 0.01                                    # N(0, 0.01)


def test_bf16_round_to_nearest_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even (1.0);
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties go to 1 + 2^-6
    v = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20, -2.5], np.float32)
    r = I.round_to_bf16(v)
    assert r.tolist() == [1.0, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7, -2.5]
    assert np.array_equal(I.round_to_bf16(r), r)
    assert np.array_equal(I.bf16_bits_to_f32(I.bf16_bits(r)), r)
    with pytest.raises(ValueError):
        I.bf16_bits(np.array([1.0 + 2.0 ** -20], np.float32))
