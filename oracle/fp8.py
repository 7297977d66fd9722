"""CPU oracle of the FP8 base product of the adapted layer.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are its only callers; the library never imports
it and it imports nothing from the library.

"Multi-LoRA Serving - S-LoRA/Punica Batching, Adapter Hot-Swap & Memory"
(the failure assumptions and "Operating it"): the base model may run in FP8
while the adapters, trained against a BF16 base, stay in BF16.  The pages fix
no quantisation recipe; the reading taken here (and by the library):

  * W is given as e4m3 codes W8 [h_out x h_in] with one fp32 scale s_w (the
    caller quantised it);
  * x (bf16) is quantised per row t: with a = amax_k |x[t][k]| (448 is
    e4m3's largest finite value), s_x[t] = a / 448 and r = 448 / a, both fp32
    divisions, and q[t][k] = e4m3(x[t][k] * r), the product in fp32, rounded
    to the nearest e4m3 value (ties to the even code), saturating at +-448;
    a row with a < 2^-120 (zeros included) takes s_x = 1 and zero codes;
  * base[t][n] = s_x[t] * s_w * sum_k q[t][k] * W8[n][k];
  * the adapter term is the bf16 one, from the unquantised x.

e4m3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
bits; exponent field 0 encodes subnormals m/8 * 2^-6; exponent 15 with
mantissa 7 is NaN (the only non-finite code), so the largest finite value is
1.75 * 2^8 = 448.

Parity status: ``e4m3_value`` pinned by exhaustive decoding properties and
``round_e4m3`` against torch's float8_e4m3fn conversion on in-range values,
plus hand-computed ties and saturation (``tests/test_fp8_oracle.py``);
``quantize_rows`` and ``base`` pinned by the exact-representation identity
(operands already on the e4m3 grid quantise to themselves, so the base equals
the plain product) and by the closed form of a one-hot row.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_value(code: int) -> float:
    """The value of one e4m3 code (NaN for the NaN codes)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _finite_table():
    """Non-negative finite e4m3 values with their codes, ascending."""
    vals = [(e4m3_value(c), c) for c in range(0x7F)]      # 0x00 .. 0x7E: +0 .. 448
    vals.sort()
    return np.array([v for v, _ in vals]), np.array([c for _, c in vals])


_VALS, _CODES = _finite_table()


def round_e4m3(v: float) -> int:
    """Code of the e4m3 value nearest to the float v (ties to the even code,
    |v| beyond 448 saturates to +-448).  v must not be NaN."""
    v = float(v)
    sign = 0x80 if (v < 0 or (v == 0 and np.signbit(v))) else 0
    a = abs(v)
    if a >= E4M3_MAX:
        return sign | 0x7E
    i = int(np.searchsorted(_VALS, a))           # first value >= a
    if _VALS[i] == a:
        return sign | int(_CODES[i])
    lo, hi = _VALS[i - 1], _VALS[i]
    dl, dh = a - lo, hi - a
    if dl < dh:
        c = _CODES[i - 1]
    elif dh < dl:
        c = _CODES[i]
    else:                                          # a tie: the even code
        c = _CODES[i - 1] if _CODES[i - 1] % 2 == 0 else _CODES[i]
    return sign | int(c)


TINY_ROW = 2.0 ** -120


def quantize_rows(x):
    """(codes uint8 [T x h], s_x float32 [T]) for bf16-valued x, in fp32."""
    x = np.asarray(x, np.float32)
    T, h = x.shape
    q = np.zeros((T, h), np.uint8)
    sx = np.ones(T, np.float32)
    for t in range(T):
        amax = np.float32(np.max(np.abs(x[t]))) if h else np.float32(0)
        if not amax >= np.float32(TINY_ROW):
            continue                                      # s_x = 1, zero codes
        sx[t] = np.float32(amax / np.float32(E4M3_MAX))   # fp32 divisions, correctly rounded
        r = np.float32(np.float32(E4M3_MAX) / amax)
        scaled = (x[t] * r).astype(np.float32)            # fp32 products, correctly rounded
        for k in range(h):
            q[t, k] = round_e4m3(scaled[k])
    return q, sx


def decode(codes):
    """float64 values of an array of e4m3 codes."""
    table = np.array([e4m3_value(c) for c in range(256)])
    return table[np.asarray(codes, np.uint8)]


def base(q, sx, W8, s_w: float, rows=None):
    """base[t][n] = s_x[t] * s_w * sum_k q[t][k] W8[n][k] in float64 for the listed rows."""
    qv = decode(q)
    Wv = decode(W8)
    rows = np.arange(qv.shape[0]) if rows is None else np.asarray(rows)
    acc = qv[rows] @ Wv.T                          # every product and partial sum exact in float64
    return acc * (np.asarray(sx, np.float64)[rows, None] * float(np.float32(s_w)))
