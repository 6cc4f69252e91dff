"""Pins of the oracle's E4M3 encoder and per-row quantisation.

The reference values come from the OCP 8-bit floating point format (E4M3:
sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals, no infinity,
S.1111.111 = NaN, max 448), decoded here independently of the oracle.
"""
import numpy as np
import pytest

import oracle
from activation_paging_gb300 import inputs


def ocp_e4m3_value(code: int) -> float:
    """Independent decoder of an E4M3 code (NaN for S.1111.111)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def enc(v):
    return int(oracle.e4m3_encode(np.array([v], np.float32))[0])


def test_known_codes():
    assert enc(448.0) == 0x7E
    assert enc(-448.0) == 0xFE
    assert enc(1.0) == 0x38
    assert enc(0.0625) == 0x18
    assert enc(0.0) == 0x00
    assert enc(-0.0) == 0x80
    assert enc(2.0 ** -9) == 0x01          # smallest subnormal
    assert enc(2.0 ** -10) == 0x00         # half of it: tie to even (zero)
    assert enc(3 * 2.0 ** -10) == 0x02     # 1.5 subnormal units: tie to even (2)
    assert enc(500.0) == 0x7E              # finite overflow saturates
    assert enc(1e30) == 0x7E and enc(-1e30) == 0xFE
    assert enc(float("inf")) == 0x7E
    assert enc(float("nan")) & 0x7F == 0x7F


def test_every_code_round_trips():
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    vals = np.array([ocp_e4m3_value(c) for c in codes], np.float32)
    got = oracle.e4m3_encode(vals)
    assert got.tolist() == codes
    for c in codes:
        assert oracle.e4m3_decode_one(c) == ocp_e4m3_value(c)


def test_midpoints_round_to_even():
    pos = [c for c in range(0x7F)]
    for c in pos[:-1]:
        lo, hi = ocp_e4m3_value(c), ocp_e4m3_value(c + 1)
        mid = (lo + hi) / 2  # exact in single precision for this format
        assert np.float32(mid) == mid
        even = c if c % 2 == 0 else c + 1
        assert enc(mid) == even, (c, mid)
        assert enc(-mid) == 0x80 | even
        assert enc(np.nextafter(np.float32(mid), np.float32(0))) == c
        assert enc(np.nextafter(np.float32(mid), np.float32(1e9))) == c + 1
    # between 448 and the would-be next value 480: saturate, never NaN
    assert enc(464.0) == 0x7E and enc(470.0) == 0x7E


def test_monotone_and_nearest_on_grid():
    g = np.linspace(-460, 460, 20001, dtype=np.float32)
    codes = oracle.e4m3_encode(g)
    vals = np.array([ocp_e4m3_value(int(c)) for c in codes])
    assert np.all(np.diff(vals) >= 0)
    table = np.array(sorted({ocp_e4m3_value(c) for c in range(256) if (c & 0x7F) != 0x7F}))
    clipped = np.clip(g.astype(np.float64), -448, 448)
    nearest_err = np.min(np.abs(table[None, :] - clipped[:, None]), axis=1)
    assert np.all(np.abs(vals - clipped) == nearest_err)


def test_quantize_rows():
    T, H = 64, 200
    x = inputs.normal_bf16(4, 0, (T, H))
    x[3] = 0          # all-zero row
    q, s = oracle.quantize_rows_e4m3(x)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    amax = np.abs(xf).max(1)
    assert s[3] == 1.0 and np.all(q[3] == 0)
    nz = amax > 0
    np.testing.assert_array_equal(s[nz], (amax[nz].astype(np.float32) / np.float32(448)))
    # the largest element maps to +-448
    for t in np.nonzero(nz)[0]:
        h = int(np.argmax(np.abs(xf[t])))
        assert q[t, h] & 0x7F == 0x7E
    # dequantised values within half a step of the format
    deq = np.vectorize(ocp_e4m3_value)(q) * s[:, None]
    err = np.abs(deq - xf)
    bound = 2.0 ** -4 * np.abs(xf) + 2.0 ** -10 * s[:, None] * 1.0001 + 1e-30
    assert np.all(err <= bound * (1 + 2 ** -20))
