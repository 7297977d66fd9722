"""Pins of the FP8 base-product oracle (no GPU): the e4m3 format decoded from
its definition, rounding checked against torch's float8_e4m3fn conversion and
hand-made ties, and the quantised product tied to the plain product where the
operands are already on the e4m3 grid."""
import numpy as np
import pytest

from oracle import fp8


def test_e4m3_decoding_properties():
    vals = [fp8.e4m3_value(c) for c in range(256)]
    nan = [c for c in range(256) if np.isnan(vals[c])]
    assert nan == [0x7F, 0xFF]
    pos = np.array(vals[:0x7F])
    assert np.all(np.diff(pos) > 0)                           # codes 0x00..0x7E ascend
    assert pos[0] == 0.0 and pos[-1] == 448.0
    assert fp8.e4m3_value(0x01) == 2.0 ** -9                   # smallest subnormal
    assert fp8.e4m3_value(0x08) == 2.0 ** -6                   # smallest normal
    assert fp8.e4m3_value(0x38) == 1.0                         # exponent field 7 = bias
    for c in range(0x7F):
        assert fp8.e4m3_value(c | 0x80) == -fp8.e4m3_value(c)


def test_every_value_rounds_to_itself_and_ties_go_to_even():
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        v = fp8.e4m3_value(c)
        got = fp8.round_e4m3(v)
        assert fp8.e4m3_value(got) == v
    vals = fp8._VALS
    for i in range(1, len(vals)):
        lo, hi = vals[i - 1], vals[i]
        mid = (lo + hi) / 2
        c = fp8.round_e4m3(mid)
        assert c % 2 == 0 and fp8.e4m3_value(c) in (lo, hi)
        assert fp8.e4m3_value(fp8.round_e4m3(np.nextafter(mid, 0))) == lo
        assert fp8.e4m3_value(fp8.round_e4m3(np.nextafter(mid, 1e9))) == hi
    # saturation (the kernel converts with satfinite)
    for v in (448.0, 449.0, 464.0, 1e6):
        assert fp8.round_e4m3(v) == 0x7E and fp8.round_e4m3(-v) == 0xFE
    assert fp8.round_e4m3(2.0 ** -11) == 0x00                 # below half the smallest subnormal


def test_rounding_agrees_with_torch_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.uniform(-448, 448, 4000), rng.normal(0, 1, 4000), rng.normal(0, 1e-2, 2000)]).astype(
        np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([fp8.round_e4m3(x) for x in v], np.uint8)
    assert np.array_equal(got, ref)


def _grid_rows(rng, T, h, scale_pow):
    """Rows of e4m3 values times 2^k whose largest magnitude is 448 * 2^k."""
    codes = rng.integers(0, 0x7E, (T, h)).astype(np.uint8) | (rng.integers(0, 2, (T, h)) * 0x80).astype(np.uint8)
    codes[:, 0] = 0x7E                                        # amax 448
    x = fp8.decode(codes) * (2.0 ** scale_pow[:, None])
    return codes, x


def test_quantization_of_grid_rows_is_exact():
    rng = np.random.default_rng(4)
    pw = rng.integers(-8, 3, 6)
    codes, x = _grid_rows(rng, 6, 40, pw)
    q, sx = fp8.quantize_rows(x.astype(np.float32))
    assert np.array_equal(sx, (2.0 ** pw).astype(np.float32))
    assert np.array_equal(fp8.decode(q), fp8.decode(codes))   # -0 and +0 decode alike
    zero = np.zeros((1, 8), np.float32)
    qz, sz = fp8.quantize_rows(zero)
    assert sz[0] == 1.0 and not qz.any()


def test_base_equals_plain_product_on_the_grid():
    rng = np.random.default_rng(5)
    pw = rng.integers(-6, 2, 9)
    codes, x = _grid_rows(rng, 9, 64, pw)
    W8 = rng.integers(0, 0x7F, (24, 64)).astype(np.uint8) | (rng.integers(0, 2, (24, 64)) * 0x80).astype(np.uint8)
    W8[W8 == 0xFF] = 0x7E
    s_w = 0.03125                                              # a power of two: every factor exact
    q, sx = fp8.quantize_rows(x.astype(np.float32))
    got = fp8.base(q, sx, W8, s_w)
    want = x @ (fp8.decode(W8) * s_w).T
    assert np.array_equal(got, want)


def test_base_one_hot_row():
    W8 = np.array([[0x38, 0x40, 0x30], [0xB8, 0x7E, 0x01]], np.uint8)   # 1, 2, 0.5 / -1, 448, 2^-9
    q = np.array([[0x00, 0x48, 0x00]], np.uint8)                          # 4 in column 1
    got = fp8.base(q, np.array([0.25], np.float32), W8, 2.0)
    assert np.array_equal(got, [[0.25 * 2.0 * 4 * 2.0, 0.25 * 2.0 * 4 * 448.0]])
