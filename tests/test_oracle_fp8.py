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


def _expected_fp8_rows(q, scale, dest, rows, fill):
    """The FP8 dispatch buffer restated with numpy: every kept pair (t, j)
    places token t's H code bytes at row dest[t, j] and its scale bits at the
    same row of the scale plane; rows no pair maps to keep the canary."""
    T, H = q.shape
    xd = np.full((rows, H), fill, np.uint8)
    xs = np.full(rows, fill * 0x01010101, np.uint32)
    tok = np.repeat(np.arange(T), dest.shape[1]).reshape(dest.shape)
    kept = dest >= 0
    xd[dest[kept]] = q[tok[kept]]
    xs[dest[kept]] = scale.view(np.uint32)[tok[kept]]
    return xd, xs


def _run_oracle_fp8(q, scale, dest, rows, fill):
    xd = np.full((rows, q.shape[1]), fill, np.uint8)
    xs = np.full(rows, fill * 0x01010101, np.uint32).view(np.float32)
    oracle.permute_rows_fp8(q, scale, dest, xd, xs)
    return xd, xs.view(np.uint32)


@pytest.mark.parametrize("T,H,k,rows,drop", [(5, 8, 2, 16, 0.0), (37, 24, 3, 200, 0.3), (64, 16, 6, 384, 0.5)])
def test_permute_rows_fp8_places_codes_and_scales(T, H, k, rows, drop):
    """Hand-built injective dest maps (some pairs dropped): the oracle's FP8
    permute matches the numpy restatement byte for byte, scales included."""
    rng = np.random.default_rng(T * 1000 + H)
    q = rng.integers(0, 256, (T, H), dtype=np.uint8)
    # distinct scales per token, so a scale taken from the wrong token or row shows
    scale = (np.arange(T, dtype=np.float32) + 1.0) * np.float32(0.375)
    dest = rng.permutation(rows)[:T * k].astype(np.int32).reshape(T, k)
    dest[rng.random((T, k)) < drop] = -1
    xd, xs = _run_oracle_fp8(q, scale, dest, rows, 0x5C)
    exd, exs = _expected_fp8_rows(q, scale, dest, rows, 0x5C)
    assert np.array_equal(xd, exd)
    assert np.array_equal(xs, exs)
    # every untouched row still holds the canary (a write past the row would show here)
    untouched = np.setdiff1d(np.arange(rows), dest[dest >= 0])
    assert np.all(xd[untouched] == 0x5C) and np.all(xs[untouched] == 0x5C5C5C5C)


def test_permute_rows_fp8_catches_swapped_scale_and_row():
    """The restatement is sharp enough to catch a plausible slip: a scale
    written for the wrong token or a code row shifted by one differ from it."""
    rng = np.random.default_rng(3)
    T, H, k, rows = 9, 8, 2, 40
    q = rng.integers(0, 256, (T, H), dtype=np.uint8)
    scale = (np.arange(T, dtype=np.float32) + 2.0)
    dest = rng.permutation(rows)[:T * k].astype(np.int32).reshape(T, k)
    exd, exs = _expected_fp8_rows(q, scale, dest, rows, 0)
    wrong_s = exs.copy()
    wrong_s[dest[0, 0]] = scale.view(np.uint32)[1]
    assert not np.array_equal(wrong_s, exs)
    wrong_x = exd.copy()
    wrong_x[dest[2, 1]] = q[3]
    assert not np.array_equal(wrong_x, exd)
    xd, xs = _run_oracle_fp8(q, scale, dest, rows, 0)
    assert np.array_equal(xd, exd) and np.array_equal(xs, exs)


def test_fp8_dispatch_padded_ragged_with_drops():
    """The whole FP8 dispatch of the oracle on a padded layout with a ragged
    expert count and drops: codes and scales are the row quantisation of each
    kept pair's token, placed at the plan's rows; padding and drops keep the
    canary."""
    T, H, E, k, C = 50, 40, 7, 3, 12   # 150 pairs into 7 x 12 rows: many drops
    x = inputs.normal_bf16(11, 0, (T, H))
    idx = np.stack([np.random.default_rng(t).choice(E, k, replace=False) for t in range(T)]).astype(np.int32)
    plan = oracle.dispatch(x, idx, E, C, True, fp8=True, fill=0x77)
    assert plan["rows"] == E * C and np.any(plan["dest"] < 0) and np.all(plan["live"] <= C)
    q, s = oracle.quantize_rows_e4m3(x)
    exd, exs = _expected_fp8_rows(q, s, plan["dest"], plan["rows"], 0x77)
    assert np.array_equal(plan["xd"], exd)
    assert np.array_equal(plan["xd_scale"].view(np.uint32), exs)
