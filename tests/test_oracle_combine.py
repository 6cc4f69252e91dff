"""Pins of the oracle's combine (top-k weighted un-permute to dense BF16)."""
import json
import os
from fractions import Fraction

import numpy as np

import oracle
from activation_paging_gb300 import inputs

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))


def bf16_ulp(v: float) -> float:
    if v == 0:
        return 2.0 ** -133
    e = np.frexp(abs(v))[1]  # v = m * 2^e, m in [0.5, 1)
    return 2.0 ** (e - 8)


def test_brute_force_exact_sum_bound():
    T, H, E, k = 40, 16, 6, 3
    idx, w = oracle.route_topk(inputs.router_logits(2, T, E), k)
    plan = oracle.dispatch_plan(idx, E, 10, True)
    y = inputs.normal_bf16(2, 2, (E * 10, H))
    out, st = oracle.combine(y, plan["dest"], w)
    assert st == 0
    yf = inputs.bf16_bits_to_f32(y)
    of = inputs.bf16_bits_to_f32(out)
    for t in range(T):
        for h in range(H):
            terms = [Fraction(float(w[t, j])) * Fraction(float(yf[plan["dest"][t, j], h]))
                     for j in range(k) if plan["dest"][t, j] >= 0]
            exact = float(sum(terms, Fraction(0)))
            mag = float(sum(abs(x) for x in terms))
            # k single-precision roundings plus the final BF16 rounding
            bound = k * 2.0 ** -24 * mag * 1.01 + 0.5 * bf16_ulp(exact) * 1.01 + 1e-38
            assert abs(float(of[t, h]) - exact) <= bound


def test_k1_unit_weight_is_a_gather():
    T, H = 33, 40
    y = inputs.normal_bf16(9, 2, (T, H))
    dest = np.random.default_rng(0).permutation(T).astype(np.int32).reshape(T, 1)
    w = np.ones((T, 1), np.float32)
    out, _ = oracle.combine(y, dest, w)
    assert np.array_equal(out, y[dest[:, 0]])


def test_all_dropped_token_is_zero():
    y = inputs.normal_bf16(1, 2, (4, 8))
    dest = np.array([[-1, -1], [0, 1], [-1, 3]], np.int32)
    w = np.full((3, 2), 0.5, np.float32)
    out, _ = oracle.combine(y, dest, w)
    assert np.all(out[0] == 0)
    yf = inputs.bf16_bits_to_f32(y)
    assert np.array_equal(out[2], inputs.f32_to_bf16_bits(np.float32(0.5) * yf[3]))


def test_identity_experts_round_trip():
    """Dispatch then combine with identity experts returns x (weights sum to 1)."""
    T, H, E, k = 128, 64, 8, 2
    idx, w = oracle.route_topk(inputs.router_logits(3, T, E), k)
    x = inputs.normal_bf16(3, 0, (T, H))
    plan = oracle.dispatch(x, idx, E, 0, False)
    out, _ = oracle.combine(plan["xd"], plan["dest"], w)
    xf, of = inputs.bf16_bits_to_f32(x), inputs.bf16_bits_to_f32(out)
    ulps = np.vectorize(bf16_ulp)(xf.astype(np.float64))
    assert np.all(np.abs(of - xf) <= ulps)


def test_out_of_range_row_is_skipped():
    y = inputs.normal_bf16(1, 2, (4, 8))
    out, st = oracle.combine(y, np.array([[1, 7]], np.int32), np.array([[1.0, 1.0]], np.float32))
    assert st & oracle.FLAG_BAD_INDEX
    assert np.array_equal(out[0], y[1])


def test_dense_output_size_golden():
    g = GOLDEN["combine_dense_output"]
    y = inputs.normal_bf16(0, 2, (4, g["hidden"]))
    dest = np.zeros((g["rows"], 1), np.int32)
    out, _ = oracle.combine(y, dest, np.ones((g["rows"], 1), np.float32))
    assert out.shape == (g["rows"], g["hidden"]) and out.nbytes == g["bytes"]
